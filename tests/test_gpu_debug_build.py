"""The -DSPEC_DEBUG variant of the library on the GPU: its kernels check the
index of every global write, of every bulk-copy range and of the partial and
candidate slots they use, and report a failed check as SPEC_DEBUG_BOUNDS in
the status word instead of faulting.  Over small cases that reach every
dispatch path (small-batch, fused, two-kernel, streaming and early-exit
samplers; greedy with one and with several blocks per row) no check may fail
and the outputs must still equal the oracle's."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from draft_verify_acceptance_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEBUG_BOUNDS = 32


@pytest.fixture(scope="module")
def dbg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from draft_verify_acceptance_gb300 import binding, build
    lib = ctypes.CDLL(build.build(debug=True))
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.spec_verify_ex.restype = I
    lib.spec_verify_ex.argtypes = [P, P, P, P, I, I, I, I, F, I, P, P, P, Z, P, P, P, P, P]
    return lib, binding


CASES = [
    # name, B, K, V, dtype, mode, recipe
    ("small_batch_f32", 8, 4, 1000, torch.float32, "sample", dict(target_std=3.0, draft_noise=0.5)),
    ("fused_f32_B200", 200, 4, 1000, torch.float32, "sample", dict(target_std=3.0, draft_noise=0.5)),
    ("fused_bf16_Kmax", 160, 64, 296, torch.bfloat16, "sample", dict(target_std=1.0, draft_noise=0.2)),
    ("two_kernel_f32", 6, 6, 20000, torch.float32, "sample", dict(target_std=5.0, independent_draft=True)),
    ("streaming_bf16_unaligned", 8, 5, 33, torch.bfloat16, "sample", dict(target_std=2.0, draft_noise=1.0)),
    ("early_exit_f32", 6, 3, 20000, torch.float32, "sample_early_exit",
     dict(target_std=5.0, independent_draft=True)),
    ("early_exit_waves_bf16", 200, 3, 32000, torch.bfloat16, "sample_early_exit",
     dict(target_std=3.0, independent_draft=True)),
    ("early_exit_two_phase_bf16", 3, 2, 400000, torch.bfloat16, "sample_early_exit",
     dict(target_std=3.0, draft_noise=0.5)),
    ("greedy_one_word", 64, 8, 3000, torch.bfloat16, "greedy", dict(target_std=4.0)),
    ("greedy_segments", 2, 2, 200000, torch.float32, "greedy", dict(target_std=4.0)),
]


@pytest.mark.parametrize("name,B,K,V,dtype,mode,recipe", CASES, ids=[c[0] for c in CASES])
def test_debug_build_checks_pass_and_outputs_match(dbg, name, B, K, V, dtype, mode, recipe):
    lib, binding = dbg
    m = binding._mode(mode)
    wmode = W.MODE_GREEDY if mode == "greedy" else W.MODE_SAMPLE
    inp = W.make_inputs(B, K, V, dtype=dtype, mode=wmode, temperature=0.9, seed=B + K + V, **recipe)
    dt = binding.DTYPE_BF16 if dtype == torch.bfloat16 else binding.DTYPE_F32
    dev = [None if t is None else t.to("cuda") for t in (inp.target, inp.draft, inp.tokens, inp.uniforms)]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsb = binding.workspace_size(B, K, V, dt, m)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    sample = m != binding.MODE_GREEDY
    rc = lib.spec_verify_ex(p(dev[0]), p(dev[1]) if sample else None, p(dev[2]),
                            p(dev[3]) if sample else None, B, K, V, dt, 0.9, m, p(acc), p(out),
                            p(ws), wsb, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                            None, None, None, p(status))
    assert rc == 0
    torch.cuda.synchronize()
    st = int(status.item())
    assert st & DEBUG_BOUNDS == 0, f"{name}: an index check failed (status {st})"
    assert st == 0, (name, st)
    assert int(ws.count_nonzero().item()) == 0
    ref = oracle.verify_ref(W.as_numpy_logits(inp.target), W.as_numpy_logits(inp.draft),
                            inp.tokens.numpy(), None if inp.uniforms is None else inp.uniforms.numpy(),
                            0.9, wmode, want_debug=True)
    ok = ref["flags"] == 0
    np.testing.assert_array_equal(acc.cpu().numpy()[ok], ref["accepted_len"][ok], err_msg=name)
    np.testing.assert_array_equal(out.cpu().numpy()[ok], ref["out_tokens"][ok], err_msg=name)
