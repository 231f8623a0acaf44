"""zero_grad_norm_noalloc: the allocation-free norm entry point, against the oracle and the
regular path.

The entry point serves callers that cannot allocate device memory (see its declaration in
include/zero_gb300.h): it keeps its scratch in a fixed array inside the library instead of
a caller-provided buffer. Here it is called through the C ABI twice in a row per case, on
two different gradient sets of a multi-bucket layout, for two rank counts, and each result
is compared with
  - the oracle's norm: the rank-ordered fp32 average of the replicas (its reduce-scatter)
    with the squares summed in fp64 (within 1e-7 relative), and the oracle's clip scale;
  - the norm and scale of a clipped zero_step on the same gradients in the recompute form,
    which runs the same norm kernel on the same grid: bit for bit.
One case clips (scale < 1) and one does not (scale exactly 1). The device memory the
process holds (torch's reserve and the driver's free bytes) is the same before and after
a call once the first call on the device has done its set-up. Pointers that are not device
memory are refused before anything is enqueued.

This file is named so that pytest collects it last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import zero_gradient_reduce_scatter_gb300 as zg
from parity_util import REL_NORM, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield


def _table(opt):
    rows = []
    for off, n, S, first in opt.buckets:
        rows += [off, n, S, first]
    return (ctypes.c_int64 * len(rows))(*rows), len(opt.buckets)


def _noalloc(grads, M, table, nb, max_norm, norm_out, scale_out, stream):
    ptrs = (ctypes.c_void_p * M)(*[g.data_ptr() for g in grads])
    return zg._lib().zero_grad_norm_noalloc(ctypes.cast(ptrs, ctypes.c_void_p), M, ctypes.cast(table, ctypes.c_void_p),
                                            nb, max_norm, norm_out, scale_out, stream)


CASES = [
    # (workload recipe, tensor sizes, M, clip threshold): the first clips, the second not
    ("1p3b", (80, 100, 20000, 5), 8, 1e-3),
    ("4b", (50, 64, 30000, 9), 4, 1e6),
]


@pytest.mark.parametrize("key,sizes,M,max_norm", CASES)
def test_noalloc_norm_matches_oracle_and_step_on_two_calls(key, sizes, M, max_norm):
    w = W.small_variant(W.workload(key), W.ragged_numel(*sizes), M=M, bucket_bytes=60000, clip=max_norm, steps=2)
    dev = torch.device("cuda")
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev), bucket_bytes=w.bucket_bytes)
    assert len(opt.buckets) > 3
    p = O.plan(w.numel, w.M, w.bucket_bytes)
    assert p.npad == opt.sizes["npad"]
    table, nb = _table(opt)
    # the regular path in the form that runs the same norm kernel on the same grid
    h = zg.Hyper(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay, clip=True,
                 max_grad_norm=max_norm, ghat_mode="recompute")
    norm_out = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    scale_out = torch.full((1,), -1.0, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    seen = []
    for k in range(2):
        grads = opt.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], opt.tensor_offsets)
        torch.cuda.synchronize()
        if k == 1:  # set-up done by the first call: this one holds no more device memory
            reserved, (free, _) = torch.cuda.memory_reserved(), torch.cuda.mem_get_info()
        rc = _noalloc(grads, w.M, table, nb, max_norm, norm_out.data_ptr(), scale_out.data_ptr(), stream)
        assert rc == 0, zg.ERRORS.get(rc, rc)
        torch.cuda.synchronize()
        if k == 1:
            assert torch.cuda.memory_reserved() == reserved
            assert torch.cuda.mem_get_info()[0] == free
        got_norm, got_scale = float(norm_out.item()), float(scale_out.item())
        # the oracle: rank-ordered fp32 average, fp64 sum of squares over real lanes
        host = [u16(g) for g in grads]
        want_norm = math.sqrt(O.global_sumsq(p, O.reduce_scatter(p, host)))
        want_scale = O.clip_scale(want_norm, max_norm)
        assert abs(got_norm - want_norm) <= REL_NORM * want_norm, (k, got_norm, want_norm)
        assert abs(got_scale - want_scale) <= 1e-6 * want_scale, (k, got_scale, want_scale)
        # the clipped step's norm and scale, bit for bit
        opt.step(grads, h)
        ref_norm, ref_scale = opt.last_norm()
        assert got_norm == ref_norm and np.float32(got_scale) == np.float32(ref_scale), (k, got_norm, ref_norm)
        if max_norm < 1.0:
            assert got_scale < 1.0, "this case must clip"
        else:
            assert got_scale == 1.0
        seen.append(got_norm)
    assert seen[0] != seen[1], "the two calls should see different gradients"


def test_noalloc_rejects_oversized_malformed_and_misplaced_arguments():
    lib = zg._lib()
    dev = torch.device("cuda")
    g = torch.zeros(64 * 2, dtype=torch.bfloat16, device=dev)
    out_n = torch.empty(1, dtype=torch.float64, device=dev)
    out_s = torch.empty(1, dtype=torch.float32, device=dev)
    ptrs = (ctypes.c_void_p * 2)(g.data_ptr(), g.data_ptr())
    nb = 2049  # one row past the fixed scratch
    rows = []
    for b in range(nb):
        rows += [0, 0, 0, b]
    big = (ctypes.c_int64 * len(rows))(*rows)
    rc = lib.zero_grad_norm_noalloc(ctypes.cast(ptrs, ctypes.c_void_p), 2, ctypes.cast(big, ctypes.c_void_p), nb,
                                    1.0, out_n.data_ptr(), out_s.data_ptr(), None)
    assert rc == -9 and b"fixed scratch" in lib.zero_strerror(rc)
    gap = (ctypes.c_int64 * 8)(0, 64, 32, 0, 100, 10, 32, 1)  # second bucket does not start at 64
    rc = lib.zero_grad_norm_noalloc(ctypes.cast(ptrs, ctypes.c_void_p), 2, ctypes.cast(gap, ctypes.c_void_p), 2,
                                    1.0, out_n.data_ptr(), out_s.data_ptr(), None)
    assert rc == -1
    huge = (ctypes.c_int64 * 4)(0, 64, 1 << 62, 0)  # M * S would overflow
    rc = lib.zero_grad_norm_noalloc(ctypes.cast(ptrs, ctypes.c_void_p), 2, ctypes.cast(huge, ctypes.c_void_p), 1,
                                    1.0, out_n.data_ptr(), out_s.data_ptr(), None)
    assert rc == -1
    ok = (ctypes.c_int64 * 4)(0, 100, 64, 0)
    host_g = torch.zeros(64 * 2, dtype=torch.bfloat16)  # pageable host memory
    host_out = torch.empty(1, dtype=torch.float64)
    mixed = (ctypes.c_void_p * 2)(g.data_ptr(), host_g.data_ptr())
    rc = lib.zero_grad_norm_noalloc(ctypes.cast(mixed, ctypes.c_void_p), 2, ctypes.cast(ok, ctypes.c_void_p), 1,
                                    1.0, out_n.data_ptr(), out_s.data_ptr(), None)
    assert rc == -1, "a host gradient pointer is refused"
    rc = lib.zero_grad_norm_noalloc(ctypes.cast(ptrs, ctypes.c_void_p), 2, ctypes.cast(ok, ctypes.c_void_p), 1,
                                    1.0, host_out.data_ptr(), out_s.data_ptr(), None)
    assert rc == -1, "a host output pointer is refused"
    rc = lib.zero_grad_norm_noalloc(ctypes.cast(ptrs, ctypes.c_void_p), 2, ctypes.cast(ok, ctypes.c_void_p), 1,
                                    1.0, out_n.data_ptr(), out_s.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert float(out_n.item()) == 0.0 and float(out_s.item()) == 1.0  # zero gradients
