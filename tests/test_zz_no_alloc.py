"""The no-allocation entry point, spec_verify_static, through the C ABI.

It serves callers that cannot allocate device memory when they verify (a
host program that only holds buffers handed to it by another runtime's
memory pool, or a decode loop in which cudaMalloc / cudaFree are not
allowed).  Its scratch is a fixed array inside the library.  These checks
compare it with spec_verify (caller-provided workspace) on two calls in a
row with different batches, and check its size limit.  This file is
collected last on purpose (pytest collects files in name order), and it
builds its own state, so it passes alone in a fresh process or after the
rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

from draft_verify_acceptance_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from draft_verify_acceptance_gb300 import binding
    return binding


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _device_inputs(inp):
    return [None if t is None else t.to("cuda") for t in
            (inp.target, inp.draft, inp.tokens, inp.uniforms)]


def _static(lib, inp, dev, stream):
    acc = torch.full((inp.B,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((inp.B, inp.K + 1), -7, dtype=torch.int32, device="cuda")
    dt = lib.DTYPE_BF16 if inp.target.dtype == torch.bfloat16 else lib.DTYPE_F32
    rc = lib._lib.spec_verify_static(_p(dev[0]), _p(dev[1]), _p(dev[2]), _p(dev[3]), inp.B,
                                     inp.K, inp.V, dt, inp.temperature, inp.mode, _p(acc),
                                     _p(out), ctypes.c_void_p(stream.cuda_stream))
    return rc, acc, out


def _with_workspace(lib, inp, dev, stream):
    acc = torch.full((inp.B,), -9, dtype=torch.int32, device="cuda")
    out = torch.full((inp.B, inp.K + 1), -9, dtype=torch.int32, device="cuda")
    dt = lib.DTYPE_BF16 if inp.target.dtype == torch.bfloat16 else lib.DTYPE_F32
    nbytes = lib.workspace_size(inp.B, inp.K, inp.V, dt, inp.mode)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    rc = lib._lib.spec_verify(_p(dev[0]), _p(dev[1]), _p(dev[2]), _p(dev[3]), inp.B, inp.K,
                              inp.V, dt, inp.temperature, inp.mode, _p(acc), _p(out), _p(ws),
                              nbytes, ctypes.c_void_p(stream.cuda_stream))
    return rc, acc, out


def test_static_scratch_matches_caller_workspace_on_two_calls_in_a_row(lib):
    stream = torch.cuda.current_stream()
    first = W.make_inputs(48, 5, 20000, dtype=torch.bfloat16, temperature=0.8, target_std=4.0,
                          draft_noise=1.0, seed=21, name="static_a")
    second = W.make_inputs(200, 8, 32000, dtype=torch.bfloat16, mode=W.MODE_GREEDY,
                           target_std=4.0, seed=22, name="static_b")
    for inp in (first, second):
        dev = _device_inputs(inp)
        rc_s, acc_s, out_s = _static(lib, inp, dev, stream)
        rc_w, acc_w, out_w = _with_workspace(lib, inp, dev, stream)
        torch.cuda.synchronize()
        assert rc_s == lib.OK and rc_w == lib.OK
        # same kernels, same arithmetic: the integer outputs agree exactly
        np.testing.assert_array_equal(acc_s.cpu().numpy(), acc_w.cpu().numpy())
        np.testing.assert_array_equal(out_s.cpu().numpy(), out_w.cpu().numpy())
        n = acc_s.cpu().numpy()
        assert ((n >= 0) & (n <= inp.K)).all()


def test_static_scratch_rejects_batches_beyond_its_size(lib):
    stream = torch.cuda.current_stream()
    B, K, V = 5000, 64, 16  # workspace of ~2.7 MB > the 1 MiB scratch
    dt = lib.DTYPE_F32
    assert lib.workspace_size(B, K, V, dt, lib.MODE_GREEDY) > lib.STATIC_SCRATCH_BYTES
    t = torch.zeros((B, K + 1, V), device="cuda")
    x = torch.zeros((B, K), dtype=torch.int32, device="cuda")
    acc = torch.full((B,), -3, dtype=torch.int32, device="cuda")
    out = torch.full((B, K + 1), -3, dtype=torch.int32, device="cuda")
    rc = lib._lib.spec_verify_static(_p(t), None, _p(x), None, B, K, V, dt, 1.0,
                                     lib.MODE_GREEDY, _p(acc), _p(out),
                                     ctypes.c_void_p(stream.cuda_stream))
    torch.cuda.synchronize()
    assert rc == lib.ERR_SCRATCH_LIMIT
    assert "scratch" in lib.status_string(rc)
    assert int(acc.min()) == -3 and int(acc.max()) == -3  # nothing was queued
