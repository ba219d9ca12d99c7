"""Parity with the oracle over seeded random shapes that cross every dispatch
rule of the library: unaligned and aligned vocabularies, rows below and above
one fused segment (4096 16-byte vectors), batches below and above one
sequence per SM, sequences that do and do not fit the small-batch kernel,
K from 0 to 64, both logit types, sampling, early-exit and greedy modes."""
import zlib

import numpy as np
import pytest
import torch

import oracle
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


def _shape(i):
    rng = np.random.default_rng(1000 + i)
    mode = ["sample", "sample", "sample_early_exit", "greedy"][i % 4]
    dtype = torch.bfloat16 if rng.random() < 0.5 else torch.float32
    V = int(rng.choice([1, 3, 17, 250, 999, 1000, 4096, 8000, 16384, 16385, 32000, 32768,
                        40000, 70001, 100000]))
    K = int(rng.choice([0, 1, 2, 4, 7, 16, 33, 64]))
    if mode == "sample_early_exit":
        K = max(K, 1)
    B = int(rng.choice([1, 3, 17, 151, 152, 153, 300]))
    # keep each case to a few hundred MB of logits at most
    esz = 2 if dtype == torch.bfloat16 else 4
    while B > 1 and B * (2 * K + 1) * V * esz > 3e8:
        B //= 2
    T = float(rng.choice([0.05, 0.5, 1.0, 1.7]))
    return mode, dtype, B, K, V, T


CASES = [_shape(i) for i in range(40)]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_random_shape_parity(lib, case):
    mode, dtype, B, K, V, T = CASES[case]
    wmode = W.MODE_GREEDY if mode == "greedy" else W.MODE_SAMPLE
    seed = zlib.crc32(repr(CASES[case]).encode()) % 1000
    inp = W.make_inputs(B, K, V, dtype=dtype, mode=wmode, temperature=T, target_std=3.0,
                        draft_noise=0.7, seed=seed)
    dev = [None if t is None else t.to("cuda") for t in (inp.target, inp.draft, inp.tokens, inp.uniforms)]
    res = lib.verify_ex(*dev, T, mode)
    torch.cuda.synchronize()
    ref = oracle.verify_ref(W.as_numpy_logits(inp.target), W.as_numpy_logits(inp.draft),
                            inp.tokens.numpy(), None if inp.uniforms is None else inp.uniforms.numpy(),
                            T, wmode, want_debug=True)
    label = f"{mode} {dtype} B={B} K={K} V={V} T={T}"
    assert int(res["status"].item()) == ref["status"] == 0, label
    n = res["accepted_len"].cpu().numpy()
    out = res["out_tokens"].cpu().numpy()
    ok = ref["flags"] == 0
    np.testing.assert_array_equal(n[ok], ref["accepted_len"][ok], err_msg=label)
    np.testing.assert_array_equal(out[ok], ref["out_tokens"][ok], err_msg=label)
    # flagged sequences are still valid outputs
    x = inp.tokens.numpy()
    for b in np.flatnonzero(~ok):
        nb = int(n[b])
        assert 0 <= nb <= K and (out[b, :nb] == x[b, :nb]).all() and 0 <= out[b, nb] < V
        assert (out[b, nb + 1:] == -1).all()
    if mode != "greedy" and K > 0:
        tol = 1e-5 if dtype == torch.float32 else 2e-3
        # early exit reports at least the positions whose rows it read: 0..n
        read = np.ones((B, K), bool)
        if mode == "sample_early_exit":
            read = np.arange(K)[None, :] <= ref["accepted_len"][:, None]
        assert np.abs(res["p_at"].cpu().numpy() - ref["p_at"])[read].max() <= tol, label
        assert np.abs(res["q_at"].cpu().numpy() - ref["q_at"])[read].max() <= tol, label
