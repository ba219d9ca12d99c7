"""Failure detection on the GPU without a fault: a bounded wait that cannot
complete must end with SPEC_DEVICE_WAIT_TIMEOUT in the status word, within
the wait limit, and leave the context usable.

The sampling kernel for rows of at most 4096 16-byte vectors decides each
sequence on one thread block, which waits until the blocks that streamed the
sequence's rows have counted them in the workspace.  Planting an arrival
count the kernel can never bring to its target (the workspace must be zero
at rest) makes that wait run out, like a flag that nothing sets.
"""
import time

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


def test_unreachable_arrival_count_times_out_and_reports(lib):
    # more sequences than SMs and short rows: the fused kernel, which is the
    # one that waits on other thread blocks
    B, K, V = 400, 4, 1000
    inp = W.make_inputs(B, K, V, dtype=torch.float32, temperature=1.0, target_std=3.0,
                        draft_noise=0.5, seed=21)
    dev = [t.to("cuda") for t in (inp.target, inp.draft, inp.tokens, inp.uniforms)]
    nbytes = lib.workspace_size(B, K, V, lib.DTYPE_F32, lib.MODE_SAMPLE)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    ws.view(torch.int32)[0] = 1 << 20  # sequence 0's arrival counter (first field of its state)
    lib.set_wait_limit(5000)  # 5 ms
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        res = lib.verify_ex(*dev, 1.0, "sample", workspace=ws)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        lib.set_wait_limit(0)
    status = int(res["status"].item())
    assert status & lib.DEVICE_WAIT_TIMEOUT, status
    assert elapsed < 0.5, elapsed  # ended within the limit (plus launch), not by a hang
    # the context is usable: a fresh workspace gives valid, oracle-equal outputs
    import oracle
    res2 = lib.verify_ex(*dev, 1.0, "sample")
    torch.cuda.synchronize()
    assert int(res2["status"].item()) == 0
    ref = oracle.verify_ref(inp.target.numpy(), inp.draft.numpy(), inp.tokens.numpy(),
                            inp.uniforms.numpy(), 1.0, oracle.MODE_SAMPLE, want_debug=True)
    ok = ref["flags"] == 0
    np.testing.assert_array_equal(res2["accepted_len"].cpu().numpy()[ok], ref["accepted_len"][ok])
    np.testing.assert_array_equal(res2["out_tokens"].cpu().numpy()[ok], ref["out_tokens"][ok])


def test_default_limit_does_not_fire_on_a_normal_call(lib):
    lib.set_wait_limit(0)
    inp = W.make_inputs(300, 4, 4000, dtype=torch.bfloat16, temperature=1.0, target_std=3.0,
                        draft_noise=0.3, seed=22)
    res = lib.verify_ex(*(t.to("cuda") for t in (inp.target, inp.draft, inp.tokens, inp.uniforms)),
                        1.0, "sample")
    torch.cuda.synchronize()
    assert int(res["status"].item()) == 0
