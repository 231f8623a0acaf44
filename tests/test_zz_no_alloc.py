"""zero_grad_norm_noalloc: the allocation-free norm entry point, against the regular path.

The entry point serves callers that cannot allocate device memory (see its declaration in
include/zero_gb300.h): it keeps its scratch in a fixed array inside the library instead of
a caller-provided buffer. Here it is called through the C ABI twice in a row, on two
different gradient sets of a multi-bucket layout, and each result is compared with the
norm and clip scale that a clipped zero_step computes for the same gradients.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import workloads as W
import zero_gradient_reduce_scatter_gb300 as zg
from parity_util import REL_NORM, make_hyper

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


def test_noalloc_norm_matches_step_norm_on_two_calls():
    w = W.small_variant(W.workload("1p3b"), W.ragged_numel(80, 100, 20000, 5), bucket_bytes=60000, clip=1.0, steps=2)
    dev = torch.device("cuda")
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, dev), bucket_bytes=w.bucket_bytes)
    assert len(opt.buckets) > 3
    table, nb = _table(opt)
    h, _ = make_hyper(w)
    norm_out = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    scale_out = torch.full((1,), -1.0, dtype=torch.float32, device=dev)
    lib = zg._lib()
    stream = torch.cuda.current_stream().cuda_stream
    seen = []
    for k in range(2):
        grads = opt.new_grad_buffers()
        for r in range(w.M):
            W.fill_grads(w, r, k, grads[r], opt.tensor_offsets)
        ptrs = (ctypes.c_void_p * w.M)(*[g.data_ptr() for g in grads])
        rc = lib.zero_grad_norm_noalloc(ctypes.cast(ptrs, ctypes.c_void_p), w.M, ctypes.cast(table, ctypes.c_void_p),
                                        nb, w.clip, norm_out.data_ptr(), scale_out.data_ptr(), stream)
        assert rc == 0, zg.ERRORS.get(rc, rc)
        opt.step(grads, h)
        ref_norm, ref_scale = opt.last_norm()
        got_norm, got_scale = float(norm_out.item()), float(scale_out.item())
        assert abs(got_norm - ref_norm) <= REL_NORM * ref_norm, (k, got_norm, ref_norm)
        assert abs(got_scale - ref_scale) <= 1e-6 * ref_scale, (k, got_scale, ref_scale)
        seen.append(got_norm)
    assert seen[0] != seen[1], "the two calls should see different gradients"


def test_noalloc_rejects_oversized_and_malformed_layouts():
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
