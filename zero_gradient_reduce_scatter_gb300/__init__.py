"""GB300-native ZeRO optimizer step: Python binding of libzero_gb300.so.

The binding only marshals arguments: every step of the path (reduce-scatter, norm and
clip, AdamW, all-gather) runs in the library's CUDA kernels. PyTorch supplies device
memory (the caller-owned buffers the C ABI borrows) and the current CUDA stream. There is
no CPU fallback: if the compiled library is missing, importing the binding's runtime fails
loudly (build it with ``__graft_entry__.build()`` or ``_build.build()``).

Typical use (one GPU, M emulated ranks)::

    import zero_gradient_reduce_scatter_gb300 as zg
    opt = zg.ZeroOptimizer(numel=[...], M=8, stage=2, master_init=w0_cuda_fp32)
    grads = opt.new_grad_buffers()              # M zeroed bf16 [npad] buffers
    opt.tensor_view(grads[r], i).copy_(g_r_i)   # rank r's gradient of tensor i
    opt.step(grads, zg.Hyper(lr=1e-3, clip=True, max_grad_norm=1.0))
    params = opt.params()                       # bf16 [n], unpadded, tensor order

The method follows "CS336 2026 Lecture 8" notes, Slides 8 and 17-26, and
"并行训练优化、MoE扩展与系统瓶颈" 1.2.2 and 2.2.1-2.2.6: reduce-scatter the gradients,
update each owner's shard with its own optimizer state, all-gather the parameters.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

# ---- constants mirrored from include/zero_gb300.h -------------------------------------
ZERO_OK = 0
ERRORS = {
    -1: "ZERO_ERR_INVALID_ARG", -2: "ZERO_ERR_MISALIGNED", -3: "ZERO_ERR_SIZE_MISMATCH",
    -4: "ZERO_ERR_STAGE", -5: "ZERO_ERR_NONFINITE", -6: "ZERO_ERR_CUDA", -7: "ZERO_ERR_BAD_CONTEXT",
    -8: "ZERO_ERR_NOT_COMPUTED", -9: "ZERO_ERR_TOO_LARGE", -10: "ZERO_ERR_DEVICE", -11: "ZERO_ERR_SCHEDULE",
}
ZERO_ERR_NONFINITE = -5
ZERO_ERR_NOT_COMPUTED = -8
ZERO_ERR_SCHEDULE = -11
ZERO_ALIGN = 64
ZERO_MAX_RANKS = 64
ZERO_MAX_SCHEDULE = 1024
GATHER = {"fused": 0, "shards": 1}
GHAT = {"auto": 0, "materialize": 1, "recompute": 2}
STATE = {"master": 0, "m": 1, "v": 2, "ghat": 3}
OVERLAP = {"none": 0, "launch": 1, "buckets": 2}
KERNELS = ("rs_norm", "norm_final", "adamw", "rs_adamw", "gather", "init", "step_begin")


class ZeroError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        text = _lib().zero_strerror(code).decode() if _LIB is not None else ""
        cuda = f" (cuda error {_LIB.zero_last_cuda_error()})" if code == -6 and _LIB is not None else ""
        super().__init__(f"{where}: {ERRORS.get(code, code)}: {text}{cuda}")


# ---- ctypes mirrors of the ABI structs --------------------------------------------------
class Config(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int32), ("stage", ctypes.c_int32), ("bucket_bytes", ctypes.c_int64),
                ("gather", ctypes.c_int32), ("groups", ctypes.c_int32), ("sharded", ctypes.c_int32),
                ("rank", ctypes.c_int32)]


class Hyper(ctypes.Structure):
    """AdamW / clipping hyper-parameters of one step (zero_hyper)."""

    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double), ("max_grad_norm", ctypes.c_double),
                ("clip", ctypes.c_int32), ("ghat_mode", ctypes.c_int32)]

    def __init__(self, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, max_grad_norm=1.0,
                 clip=False, ghat_mode="auto"):
        super().__init__(lr, beta1, beta2, eps, weight_decay, max_grad_norm, 1 if clip else 0, GHAT[ghat_mode])


class Sizes(ctypes.Structure):
    _fields_ = [(k, ctypes.c_int64) for k in (
        "npad", "n", "n_buckets", "shard_len", "bytes_master", "bytes_m", "bytes_v", "bytes_ghat",
        "bytes_param_full", "bytes_param_shards", "bytes_grad_each", "bytes_scratch")]


class Buffers(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in ("master", "m", "v", "ghat", "param_full", "param_shards", "scratch")]


# ---- library loading -------------------------------------------------------------------
_LIB = None
_LOCK = threading.Lock()
_P, _I32, _I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64

# name -> (restype, argtypes); every function declared in include/zero_gb300.h
SIGNATURES = {
    "zero_plan": (ctypes.c_int, [ctypes.POINTER(Config), _P, _I64, ctypes.POINTER(Sizes)]),
    "zero_plan_layout": (ctypes.c_int, [ctypes.POINTER(Config), _P, _I64, _P, _P]),
    "zero_init": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.POINTER(Config), _P, _I64, ctypes.POINTER(Buffers),
                                 _P, _P]),
    "zero_step": (ctypes.c_int, [_P, _P, ctypes.c_int, ctypes.POINTER(Hyper), _P]),
    "zero_step_host": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, ctypes.POINTER(Hyper), _P, _P]),
    "zero_step_host_overlapped": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, ctypes.POINTER(Hyper), _P, _P, _P]),
    "zero_reduce_bucket": (ctypes.c_int, [_P, _I64, _P, _P]),
    "zero_apply": (ctypes.c_int, [_P, ctypes.c_int, ctypes.POINTER(Hyper), _P]),
    "zero_step_bucket": (ctypes.c_int, [_P, ctypes.c_int64, _P, ctypes.c_int, ctypes.POINTER(Hyper), _P]),
    "zero_step_bucket_scheduled": (ctypes.c_int, [_P, ctypes.c_int64, _P, ctypes.c_int, _P]),
    "zero_set_schedule": (ctypes.c_int, [_P, _P, ctypes.c_int64, _P]),
    "zero_step_scheduled": (ctypes.c_int, [_P, _P, ctypes.c_int, _P]),
    "zero_apply_scheduled": (ctypes.c_int, [_P, ctypes.c_int, _P]),
    "zero_params": (ctypes.c_int, [_P, ctypes.POINTER(_P)]),
    "zero_save_state": (ctypes.c_int, [_P, _P, _P, _P, _P]),
    "zero_load_state": (ctypes.c_int, [_P, _P, _P, _P, _I64, _P]),
    "zero_gather": (ctypes.c_int, [_P, _I64, _P, _P]),
    "zero_gather_bucket": (ctypes.c_int, [_P, _I64, _P, _P]),
    "zero_bucket_info": (ctypes.c_int, [_P, _I64, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "zero_get_state": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, _P, _P]),
    "zero_last_norm": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_float)]),
    "zero_sync_status": (ctypes.c_int, [_P]),
    "zero_check_report": (ctypes.c_int, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "zero_checked_build": (ctypes.c_int, []),
    "zero_get_step": (ctypes.c_int, [_P, ctypes.POINTER(_I64)]),
    "zero_set_step": (ctypes.c_int, [_P, _I64]),
    "zero_set_timing": (ctypes.c_int, [_P, ctypes.c_int]),
    "zero_kernel_times": (ctypes.c_int, [_P, _P, _P]),
    "zero_launch_shape": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "zero_set_max_ctas": (ctypes.c_int, [_P, ctypes.c_int]),
    "zero_set_launch_overlap": (ctypes.c_int, [_P, ctypes.c_int]),
    "zero_destroy": (ctypes.c_int, [_P]),
    "zero_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "zero_last_cuda_error": (ctypes.c_int, []),
    "zero_state_bytes_per_param": (ctypes.c_double, [ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                     ctypes.c_double, ctypes.c_double]),
    "zero_grad_norm_noalloc": (ctypes.c_int, [_P, ctypes.c_int, _P, _I64, ctypes.c_double, _P, _P, _P]),
    "zero_rank_step": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, ctypes.POINTER(Hyper), _P]),
    "zero_rank_sumsq": (ctypes.c_int, [_P, _P, ctypes.POINTER(Hyper), _P, _P]),
    "zero_rank_partial": (ctypes.c_int, [_P, _P, _P, _P]),
    "zero_rank_partial_bucket": (ctypes.c_int, [_P, ctypes.c_int64, _P, _P, _P]),
    "zero_rank_step_bucket": (ctypes.c_int, [_P, _I64, _P, ctypes.c_int, ctypes.POINTER(Hyper), _P]),
    "zero_rank_reduce_bucket": (ctypes.c_int, [_P, _I64, _P, _P]),
}


def library_path() -> str:
    return _build.LIB_PATH


def _lib():
    """Loads libzero_gb300.so; raises if it has not been built (no fallback exists)."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build the CUDA library first "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _LIB = lib
    return _LIB


def _check(code: int, where: str):
    if code != ZERO_OK:
        raise ZeroError(code, where)


def _i64_array(vals):
    arr = (ctypes.c_int64 * max(len(vals), 1))(*[int(v) for v in vals])
    return arr


# The current stream's raw handle without building a torch.cuda.Stream object (the getter
# torch's own generated code uses; ~0.3 us against ~3 us, which matters for steps of a few
# microseconds); the public path when this torch lacks it.
_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_CUR_DEVICE = getattr(torch._C, "_cuda_getDevice", None)


def _stream_handle(stream) -> int:
    if stream is not None:
        return int(stream.cuda_stream)
    if _RAW_STREAM is not None and _CUR_DEVICE is not None:
        return int(_RAW_STREAM(_CUR_DEVICE()))
    return int(torch.cuda.current_stream().cuda_stream)


# ---- host-only planning -----------------------------------------------------------------
def plan(numel, M: int, stage: int, bucket_bytes: int = 0, gather: str = "fused", groups: int = 1,
         rank: int | None = None) -> dict:
    """Layout sizes of the ZeRO step (host only, no CUDA). rank: the sizes of one rank of the
    process-per-rank mode (its shard of the state) instead of the emulated job's."""
    cfg = Config(M, stage, bucket_bytes, GATHER[gather], groups if groups > 1 else 0,
                 0 if rank is None else 1, rank or 0)
    arr = _i64_array(numel)
    out = Sizes()
    _check(_lib().zero_plan(ctypes.byref(cfg), ctypes.cast(arr, _P), len(numel), ctypes.byref(out)), "zero_plan")
    return {k: getattr(out, k) for k, _ in Sizes._fields_}


def layout(numel, M: int, stage: int, bucket_bytes: int = 0, gather: str = "fused", groups: int = 1):
    """(tensor_offsets, buckets): padded start lane of each tensor and, per bucket,
    (off, n, S, first_tensor)."""
    sizes = plan(numel, M, stage, bucket_bytes, gather, groups)
    cfg = Config(M, stage, bucket_bytes, GATHER[gather], groups if groups > 1 else 0)
    arr = _i64_array(numel)
    toff = (ctypes.c_int64 * max(len(numel), 1))()
    btab = (ctypes.c_int64 * max(4 * sizes["n_buckets"], 1))()
    _check(_lib().zero_plan_layout(ctypes.byref(cfg), ctypes.cast(arr, _P), len(numel), ctypes.cast(toff, _P),
                                   ctypes.cast(btab, _P)), "zero_plan_layout")
    buckets = [tuple(btab[4 * b:4 * b + 4]) for b in range(sizes["n_buckets"])]
    return list(toff[:len(numel)]), buckets


def state_bytes_per_param(stage: int, M: int, param_bytes: float, grad_bytes: float, optim_bytes: float) -> float:
    return _lib().zero_state_bytes_per_param(stage, M, param_bytes, grad_bytes, optim_bytes)


# ---- the optimizer -----------------------------------------------------------------------
class ZeroOptimizer:
    """M emulated data-parallel ranks on one GPU; one ``step`` = one ZeRO optimizer step.

    Buffers (fp32 master / m / v in the padded owner-sharded layout, the unpadded bf16
    parameters, optional fp32 averaged-gradient workspace, optional bf16 shards, scratch)
    are allocated here with torch and lent to the C context.
    """

    def __init__(self, numel, M: int, stage: int, master_init: torch.Tensor, bucket_bytes: int = 0,
                 gather: str = "fused", ghat_buffer: bool | None = None, stream=None, groups: int = 1):
        if not (isinstance(master_init, torch.Tensor) and master_init.is_cuda and master_init.dtype == torch.float32):
            raise TypeError("master_init must be a CUDA float32 tensor of the unpadded parameters")
        self.numel = [int(x) for x in numel]
        self.M, self.stage, self.bucket_bytes, self.gather = int(M), int(stage), int(bucket_bytes), gather
        self.groups = max(1, int(groups))
        self.K = self.M // self.groups  # owners sharing one copy of the state
        self.sizes = plan(self.numel, M, stage, bucket_bytes, gather, self.groups)
        self.tensor_offsets, self.buckets = layout(self.numel, M, stage, bucket_bytes, gather, self.groups)
        s = self.sizes
        if master_init.numel() != s["n"]:
            raise ValueError(f"master_init has {master_init.numel()} values, the tensors {s['n']}")
        dev = master_init.device
        self.device = dev
        npad = s["npad"]
        self.master = torch.empty(npad, dtype=torch.float32, device=dev)
        self.m = torch.empty(npad, dtype=torch.float32, device=dev)
        self.v = torch.empty(npad, dtype=torch.float32, device=dev)
        # The averaged-gradient workspace pays off when clipping with M > 4 (see ZERO_GHAT_AUTO).
        if ghat_buffer is None:
            ghat_buffer = M > 4
        self.ghat = torch.empty(npad, dtype=torch.float32, device=dev) if ghat_buffer else None
        self.param_full = torch.empty(s["n"], dtype=torch.bfloat16, device=dev)
        self.param_shards = (torch.empty(npad, dtype=torch.bfloat16, device=dev)
                             if gather == "shards" else None)
        self.scratch = torch.empty(s["bytes_scratch"], dtype=torch.uint8, device=dev)
        bufs = Buffers(self.master.data_ptr(), self.m.data_ptr(), self.v.data_ptr(),
                       self.ghat.data_ptr() if self.ghat is not None else None, self.param_full.data_ptr(),
                       self.param_shards.data_ptr() if self.param_shards is not None else None,
                       self.scratch.data_ptr())
        cfg = Config(M, stage, bucket_bytes, GATHER[gather], self.groups if self.groups > 1 else 0)
        arr = _i64_array(self.numel)
        ctx = _P()
        mi = master_init.contiguous()
        _check(_lib().zero_init(ctypes.byref(ctx), ctypes.byref(cfg), ctypes.cast(arr, _P), len(self.numel),
                                ctypes.byref(bufs), mi.data_ptr(), _stream_handle(stream)), "zero_init")
        self._ctx = ctx
        self._grad_ptrs = (ctypes.c_void_p * M)()

    # -- gradients ------------------------------------------------------------------------
    def new_grad_buffers(self):
        """M zeroed bf16 gradient buffers in the padded layout."""
        return [torch.zeros(self.sizes["npad"], dtype=torch.bfloat16, device=self.device) for _ in range(self.M)]

    def tensor_view(self, buf: torch.Tensor, i: int) -> torch.Tensor:
        """View of tensor i inside a padded flat buffer (gradient or state)."""
        o = self.tensor_offsets[i]
        return buf[o:o + self.numel[i]]

    # -- the step ---------------------------------------------------------------------------
    def _ptrs(self, grads):
        if len(grads) != self.M:
            raise ValueError(f"expected {self.M} gradient buffers, got {len(grads)}")
        for r, g in enumerate(grads):
            if not (g.is_cuda and g.dtype == torch.bfloat16 and g.is_contiguous() and g.numel() == self.sizes["npad"]):
                raise ValueError(f"grads[{r}] must be a contiguous CUDA bf16 tensor of npad={self.sizes['npad']}")
            self._grad_ptrs[r] = g.data_ptr()
        return self._grad_ptrs

    def step(self, grads, hyper: Hyper, stage: int | None = None, stream=None):
        ptrs = self._ptrs(grads)
        _check(_lib().zero_step(self._ctx, ctypes.cast(ptrs, _P), self.stage if stage is None else stage,
                                ctypes.byref(hyper), _stream_handle(stream)), "zero_step")

    def step_host(self, host_grads, dev_grads, host_params: torch.Tensor, hyper: Hyper, stream=None):
        """Step from pinned host gradients; the updated bf16 parameters land in host_params."""
        for g in host_grads:
            if g.is_cuda or g.dtype != torch.bfloat16 or g.numel() != self.sizes["npad"]:
                raise ValueError("host_grads must be pinned host bf16 tensors of npad elements")
        if host_params.is_cuda or host_params.numel() != self.sizes["n"]:
            raise ValueError("host_params must be a pinned host bf16 tensor of n elements")
        hp = (ctypes.c_void_p * self.M)(*[g.data_ptr() for g in host_grads])
        dp = self._ptrs(dev_grads)
        _check(_lib().zero_step_host(self._ctx, ctypes.cast(hp, _P), ctypes.cast(dp, _P), self.stage,
                                     ctypes.byref(hyper), host_params.data_ptr(), _stream_handle(stream)),
               "zero_step_host")

    # -- ZeRO-2 per-bucket streaming ----------------------------------------------------------
    def bucket_lanes(self, bucket: int) -> int:
        off, n, S, _ = self.buckets[bucket]
        return self.K * S

    def new_bucket_grad_buffers(self, bucket: int):
        """M zeroed bf16 buffers for one bucket (M * S_b lanes each)."""
        return [torch.zeros(self.bucket_lanes(bucket), dtype=torch.bfloat16, device=self.device)
                for _ in range(self.M)]

    def bucket_tensor_view(self, bucket_buf: torch.Tensor, bucket: int, i: int) -> torch.Tensor:
        """View of tensor i (which must live in `bucket`) inside a bucket gradient buffer."""
        off = self.buckets[bucket][0]
        o = self.tensor_offsets[i] - off
        if not (0 <= o and o + self.numel[i] <= self.bucket_lanes(bucket)):
            raise ValueError(f"tensor {i} is not in bucket {bucket}")
        return bucket_buf[o:o + self.numel[i]]

    def _bucket_ptrs(self, bucket: int, grads_b):
        if len(grads_b) != self.M:
            raise ValueError(f"expected {self.M} bucket gradient buffers")
        lanes = self.bucket_lanes(bucket)
        for g in grads_b:
            if not (g.is_cuda and g.dtype == torch.bfloat16 and g.is_contiguous() and g.numel() >= lanes):
                raise ValueError("bucket gradients must be contiguous CUDA bf16 tensors of M * S_b lanes")
        return (ctypes.c_void_p * self.M)(*[g.data_ptr() for g in grads_b])

    def reduce_bucket(self, bucket: int, grads_b, stream=None):
        ptrs = self._bucket_ptrs(bucket, grads_b)
        _check(_lib().zero_reduce_bucket(self._ctx, bucket, ctypes.cast(ptrs, _P), _stream_handle(stream)),
               "zero_reduce_bucket")

    def step_bucket(self, bucket: int, grads_b, hyper: Hyper, stream=None):
        """ZeRO-2 without clipping: reduce-scatter and update bucket `bucket` in one pass; the
        step completes (t advances) once every bucket has been stepped."""
        ptrs = self._bucket_ptrs(bucket, grads_b)
        _check(_lib().zero_step_bucket(self._ctx, bucket, ctypes.cast(ptrs, _P), self.stage, ctypes.byref(hyper),
                                       _stream_handle(stream)), "zero_step_bucket")

    def apply(self, hyper: Hyper, stream=None):
        _check(_lib().zero_apply(self._ctx, self.stage, ctypes.byref(hyper), _stream_handle(stream)), "zero_apply")

    # ---- steps with device-resident scalars (CUDA graph capture) ----------------------
    def set_schedule(self, hypers, stream=None):
        """Upload the hyper-parameters of the next len(hypers) steps (one Hyper each; equal
        clip and ghat_mode) to the device; None or [] leaves scheduled mode. Synchronises."""
        hypers = list(hypers or [])
        arr = (Hyper * len(hypers))(*hypers) if hypers else None
        _check(_lib().zero_set_schedule(self._ctx, ctypes.cast(arr, _P) if arr is not None else None, len(hypers),
                                        _stream_handle(stream)), "zero_set_schedule")

    def step_scheduled(self, grads, stream=None):
        """step() with this step's hyper-parameters taken from the device schedule; only
        kernel launches, so it can be captured in a CUDA graph (each replay is a step)."""
        ptrs = self._ptrs(grads)
        _check(_lib().zero_step_scheduled(self._ctx, ctypes.cast(ptrs, _P), self.stage, _stream_handle(stream)),
               "zero_step_scheduled")

    def step_bucket_scheduled(self, bucket: int, grads_b, stream=None):
        """step_bucket() with this step's hyper-parameters taken from the device schedule."""
        ptrs = self._bucket_ptrs(bucket, grads_b)
        _check(_lib().zero_step_bucket_scheduled(self._ctx, bucket, ctypes.cast(ptrs, _P), self.stage,
                                                 _stream_handle(stream)), "zero_step_bucket_scheduled")

    def apply_scheduled(self, stream=None):
        """apply() with this step's hyper-parameters taken from the device schedule."""
        _check(_lib().zero_apply_scheduled(self._ctx, self.stage, _stream_handle(stream)), "zero_apply_scheduled")

    def step_host_overlapped(self, host_grads, dev_grads, host_params: torch.Tensor, hyper: Hyper,
                             copy_stream, stream=None):
        """step_host with the host-to-device copies on `copy_stream`, overlapping the previous
        step's kernels and parameter copy when dev_grads alternates between two sets."""
        for g in host_grads:
            if g.is_cuda or g.dtype != torch.bfloat16 or g.numel() != self.sizes["npad"]:
                raise ValueError("host_grads must be pinned host bf16 tensors of npad elements")
        if host_params.is_cuda or host_params.numel() != self.sizes["n"]:
            raise ValueError("host_params must be a pinned host bf16 tensor of n elements")
        hp = (ctypes.c_void_p * self.M)(*[g.data_ptr() for g in host_grads])
        dp = (ctypes.c_void_p * self.M)(*[g.data_ptr() for g in dev_grads])
        for g in dev_grads:
            if not (g.is_cuda and g.dtype == torch.bfloat16 and g.numel() == self.sizes["npad"]):
                raise ValueError("dev_grads must be CUDA bf16 tensors of npad elements")
        _check(_lib().zero_step_host_overlapped(self._ctx, ctypes.cast(hp, _P), ctypes.cast(dp, _P), self.stage,
                                                ctypes.byref(hyper), host_params.data_ptr(), _stream_handle(stream),
                                                int(copy_stream.cuda_stream)), "zero_step_host_overlapped")

    def gather_params(self, bucket: int = -1, dst: torch.Tensor | None = None, stream=None):
        _check(_lib().zero_gather(self._ctx, bucket, dst.data_ptr() if dst is not None else None,
                                  _stream_handle(stream)), "zero_gather")

    def gather_bucket(self, bucket: int, dst: torch.Tensor, stream=None):
        """ZeRO-3: bucket `bucket`'s bf16 parameters into the transient buffer dst[:n_b]."""
        if not (dst.is_cuda and dst.dtype == torch.bfloat16 and dst.numel() >= self.buckets[bucket][1]):
            raise ValueError("dst must be a CUDA bf16 tensor with room for the bucket")
        _check(_lib().zero_gather_bucket(self._ctx, bucket, dst.data_ptr(), _stream_handle(stream)),
               "zero_gather_bucket")

    def bucket_range(self, bucket: int):
        """(first unpadded index, parameter count) of a bucket."""
        u, n = _I64(), _I64()
        _check(_lib().zero_bucket_info(self._ctx, bucket, ctypes.byref(u), ctypes.byref(n)), "zero_bucket_info")
        return u.value, n.value

    def _side_streams(self, count: int, exclude) -> list:
        """`count` distinct side streams kept by this optimizer (made once, reused by later
        calls), none of them the same CUDA stream as any in `exclude`."""
        if count <= 0:
            return []
        taken = {int(x.cuda_stream) for x in exclude}
        pool = getattr(self, "_prefetch_streams", None)
        if pool is None:
            pool = self._prefetch_streams = []
        out = []
        for x in pool:
            if len(out) < count and int(x.cuda_stream) not in taken:
                out.append(x)
                taken.add(int(x.cuda_stream))
        for _ in range(64):  # torch hands out pool streams in turn; skip ones already taken
            if len(out) == count:
                break
            x = torch.cuda.Stream(device=self.device)
            if int(x.cuda_stream) not in taken and all(int(x.cuda_stream) != int(y.cuda_stream) for y in pool):
                pool.append(x)
                out.append(x)
                taken.add(int(x.cuda_stream))
        if len(out) < count:
            raise RuntimeError(f"could not find {count} distinct side streams")
        return out

    def prefetched_buckets(self, order, stream=None, side_stream=None, buffers: int = 4):
        """ZeRO-3 just-in-time parameters with prefetch.

        Yields (bucket, params) in `order`; `params` (bf16, the bucket's n_b values) is ready
        for work queued on `stream` when yielded. The gathers of the next `buffers - 1`
        buckets run on side streams meanwhile, each into a transient buffer of its own
        (`buffers` of them, used in turn); a buffer is reused only after the work the consumer
        queued on `stream` while it held that buffer has finished with it. Each buffer has a
        side stream of its own (`side_stream` may be one stream or a sequence; missing ones
        are made), so consecutive gathers do not wait for each other: each waits only for its
        buffer's last consumer, and another buffer's gather runs while it waits.
        The default of four buffers is the measured best on GB300: a 129-bucket sweep of the
        4B layout took 2.39 ms with four (101.5% of the copy peak, the gather kernels' own
        time) against 2.58 ms with two and 2.54 with three; six gave no more. The transient
        memory is `buffers` times the largest bucket.
        """
        order = list(order)
        if not order:
            return
        if buffers < 2:
            raise ValueError("buffers must be at least 2")
        stream = stream or torch.cuda.current_stream()
        if isinstance(side_stream, (tuple, list)):
            sides = list(side_stream)
        else:
            sides = [side_stream] if side_stream is not None else []
        sides += self._side_streams(buffers - len(sides), exclude=[stream] + sides)
        cap = max(self.buckets[b][1] for b in order)
        bufs = [torch.empty(cap, dtype=torch.bfloat16, device=self.device) for _ in range(buffers)]
        ready = [torch.cuda.Event() for _ in range(buffers)]
        free = [torch.cuda.Event() for _ in range(buffers)]
        for i in range(buffers):
            free[i].record(stream)

        def issue(i):
            slot = i % buffers
            sides[slot].wait_event(free[slot])
            self.gather_bucket(order[i], bufs[slot], stream=sides[slot])
            ready[slot].record(sides[slot])

        for i in range(min(buffers - 1, len(order))):
            issue(i)
        for i, b in enumerate(order):
            if i + buffers - 1 < len(order):
                issue(i + buffers - 1)
            slot = i % buffers
            stream.wait_event(ready[slot])
            yield b, bufs[slot][:self.buckets[b][1]]
            free[slot].record(stream)

    # -- results ------------------------------------------------------------------------------
    def params(self) -> torch.Tensor:
        ptr = _P()
        _check(_lib().zero_params(self._ctx, ctypes.byref(ptr)), "zero_params")
        assert ptr.value == self.param_full.data_ptr()
        return self.param_full

    def get_state(self, which: str, rank: int, stream=None) -> torch.Tensor:
        out = torch.empty(self.sizes["shard_len"], dtype=torch.float32, device=self.device)
        _check(_lib().zero_get_state(self._ctx, STATE[which], rank, out.data_ptr(), _stream_handle(stream)),
               "zero_get_state")
        return out

    # -- checkpoint / resume / reshard ---------------------------------------------------------
    def save_state(self, stream=None) -> dict:
        """Layout-independent state: unpadded fp32 master / m / v (device tensors) and t."""
        n = self.sizes["n"]
        out = {k: torch.empty(n, dtype=torch.float32, device=self.device) for k in ("master", "m", "v")}
        _check(_lib().zero_save_state(self._ctx, out["master"].data_ptr(), out["m"].data_ptr(), out["v"].data_ptr(),
                                      _stream_handle(stream)), "zero_save_state")
        out["t"] = self.t
        return out

    def load_state(self, state: dict, stream=None):
        """Loads a state saved by any context over the same tensors (any M, bucket size, stage)."""
        n = self.sizes["n"]
        ts = {}
        for k in ("master", "m", "v"):
            x = state.get(k)
            if x is not None:
                x = x.to(device=self.device, dtype=torch.float32).contiguous()
                if x.numel() != n:
                    raise ValueError(f"{k} has {x.numel()} values, expected {n}")
            ts[k] = x
        if ts["master"] is None:
            raise ValueError("state needs the master weights")
        _check(_lib().zero_load_state(self._ctx, ts["master"].data_ptr(),
                                      ts["m"].data_ptr() if ts["m"] is not None else None,
                                      ts["v"].data_ptr() if ts["v"] is not None else None, int(state.get("t", 0)),
                                      _stream_handle(stream)), "zero_load_state")
        (stream or torch.cuda.current_stream()).synchronize()  # the inputs may be temporaries

    def state_dict(self) -> dict:
        """Host copy for a checkpoint file (torch.save-able), with the tensor sizes."""
        st = self.save_state()
        torch.cuda.current_stream().synchronize()
        return {"numel": list(self.numel), "t": st["t"], **{k: st[k].cpu() for k in ("master", "m", "v")}}

    def load_state_dict(self, sd: dict):
        if list(sd["numel"]) != list(self.numel):
            raise ValueError("checkpoint was written for different tensors")
        self.load_state(sd)

    def last_norm(self):
        """(norm, scale) of the last clipped step, or None if it did not clip."""
        n, s = ctypes.c_double(), ctypes.c_float()
        rc = _lib().zero_last_norm(self._ctx, ctypes.byref(n), ctypes.byref(s))
        if rc == ZERO_ERR_NOT_COMPUTED:
            return None
        _check(rc, "zero_last_norm")
        return n.value, s.value

    def sync_status(self) -> int:
        """0, ZERO_ERR_NONFINITE if the last clipped step was skipped, or ZERO_ERR_SCHEDULE if
        a scheduled step found no schedule entry."""
        rc = _lib().zero_sync_status(self._ctx)
        if rc not in (ZERO_OK, ZERO_ERR_NONFINITE, ZERO_ERR_SCHEDULE):
            _check(rc, "zero_sync_status")
        return rc

    def check_report(self):
        """(site, index) of the first failed bounds check of a checked build; site 0 = none."""
        site, idx = _I64(), _I64()
        _check(_lib().zero_check_report(self._ctx, ctypes.byref(site), ctypes.byref(idx)), "zero_check_report")
        return site.value, idx.value

    @property
    def t(self) -> int:
        t = ctypes.c_int64()
        _check(_lib().zero_get_step(self._ctx, ctypes.byref(t)), "zero_get_step")
        return t.value

    @t.setter
    def t(self, value: int):
        _check(_lib().zero_set_step(self._ctx, int(value)), "zero_set_step")

    def set_timing(self, on: bool):
        _check(_lib().zero_set_timing(self._ctx, 1 if on else 0), "zero_set_timing")

    def kernel_times(self) -> dict:
        """{kernel: (total ms, launches)} since the previous call (timing must be on)."""
        ms = (ctypes.c_double * len(KERNELS))()
        cnt = (ctypes.c_int64 * len(KERNELS))()
        _check(_lib().zero_kernel_times(self._ctx, ctypes.cast(ms, _P), ctypes.cast(cnt, _P)), "zero_kernel_times")
        return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNELS)}

    def launch_shape(self):
        ctas, thr = ctypes.c_int(), ctypes.c_int()
        _check(_lib().zero_launch_shape(self._ctx, ctypes.byref(ctas), ctypes.byref(thr)), "zero_launch_shape")
        return ctas.value, thr.value

    def set_launch_overlap(self, mode: str):
        """Programmatic launch overlap of the per-bucket kernels: "none", "launch" (each waits
        for its predecessor before touching memory) or "buckets" (consecutive per-bucket
        launches of this optimizer on one stream overlap; see zero_set_launch_overlap)."""
        _check(_lib().zero_set_launch_overlap(self._ctx, OVERLAP[mode]), "zero_set_launch_overlap")

    def set_max_ctas(self, ctas: int):
        """Cap the grid of the streaming kernels (0 = none); for testing index arithmetic."""
        _check(_lib().zero_set_max_ctas(self._ctx, int(ctas)), "zero_set_max_ctas")

    def close(self):
        if getattr(self, "_ctx", None) is not None and self._ctx.value:
            _lib().zero_destroy(self._ctx)
            self._ctx = _P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# process-per-rank mode (one process per GPU); imported last: it builds on the names above
from .sharded import ShardedZeroOptimizer  # noqa: E402
