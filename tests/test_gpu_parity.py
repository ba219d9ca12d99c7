"""Parity of the CUDA verify path (through the C ABI) with the CPU oracle.

Bar (per sequence):
  greedy   accepted_len and out_tokens bit-equal, always;
  sampling accepted_len and out_tokens bit-equal for every sequence the
           oracle does not flag as a boundary case (a uniform within 1e-6 of
           an accept ratio or of a CDF step, or a residual mass below 1e-6);
           flagged sequences are counted and must still be valid outputs;
  p_i(x_i), q_i(x_i) within 1e-5 absolute (fp32 logits) or 2e-3 (bf16);
  the device status word equals the oracle's data-error bits.
"""
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


def _dev(t):
    return None if t is None else t.to("cuda")


# Canary guards: every output, the status word and the workspace sit inside a
# larger buffer whose GUARD bytes on each side hold the byte CANARY; after the
# call every guard byte must still hold it (an out-of-range write by any
# kernel shows up here), and the workspace body must be back to all zeros.
GUARD = 256
CANARY = 0xA5


class Guarded:
    def __init__(self, shape, dtype, fill=None):
        self.shape, self.dtype = tuple(shape), dtype
        self.nbytes = int(np.prod(self.shape, dtype=np.int64)) * torch.empty(0, dtype=dtype).element_size()
        self.buf = torch.full((self.nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        if fill is not None:
            self.buf[GUARD:GUARD + self.nbytes].fill_(fill)
        self.body = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(self.shape)

    def ptr(self):
        import ctypes
        return ctypes.c_void_p(self.buf.data_ptr() + GUARD)

    def guards_intact(self):
        g = torch.cat([self.buf[:GUARD], self.buf[GUARD + self.nbytes:]])
        return bool((g == CANARY).all().item())


def run_gpu_mode(lib, inp, mode):
    """spec_verify_ex through the C ABI with every output, the status word and
    the workspace in guarded buffers; fails if a guard byte changed or the
    workspace is not left zero-filled."""
    import ctypes
    mode = lib._mode(mode)
    B, K, V = inp.B, inp.K, inp.V
    dt = lib.DTYPE_BF16 if inp.target.dtype == torch.bfloat16 else lib.DTYPE_F32
    dev = [_dev(t) for t in (inp.target, inp.draft, inp.tokens, inp.uniforms)]
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    acc = Guarded((B,), torch.int32)
    out = Guarded((B, K + 1), torch.int32)
    p_at = Guarded((B, K), torch.float32, 0)
    q_at = Guarded((B, K), torch.float32, 0)
    flags = Guarded((B,), torch.int32, 0)
    status = Guarded((1,), torch.int32, 0)
    wsb = lib.workspace_size(B, K, V, dt, mode)
    ws = Guarded((wsb,), torch.uint8, 0)
    sample = mode != lib.MODE_GREEDY
    stream = torch.cuda.current_stream()
    rc = lib._lib.spec_verify_ex(
        ptr(dev[0]), ptr(dev[1]) if sample else None, ptr(dev[2]) if K > 0 else None,
        ptr(dev[3]) if sample else None, B, K, V, dt, float(inp.temperature), mode,
        acc.ptr(), out.ptr(), ws.ptr(), wsb, ctypes.c_void_p(stream.cuda_stream),
        p_at.ptr(), q_at.ptr(), flags.ptr(), status.ptr())
    assert rc == lib.OK, lib.status_string(rc)
    torch.cuda.synchronize()
    for name, g in (("accepted_len", acc), ("out_tokens", out), ("p_at", p_at), ("q_at", q_at),
                    ("flags", flags), ("status", status), ("workspace", ws)):
        assert g.guards_intact(), f"a kernel wrote outside {name}"
    if int(status.body.item()) == 0:
        assert int(ws.body.count_nonzero().item()) == 0, "workspace not left zero-filled"
    return {"accepted_len": acc.body.cpu().numpy(), "out_tokens": out.body.cpu().numpy(),
            "p_at": p_at.body.cpu().numpy(), "q_at": q_at.body.cpu().numpy(),
            "flags": flags.body.cpu().numpy(), "status": status.body.cpu().numpy()}


def run_gpu(lib, inp):
    return run_gpu_mode(lib, inp, inp.mode)


def run_oracle(inp):
    return oracle.verify_ref(W.as_numpy_logits(inp.target), W.as_numpy_logits(inp.draft),
                             inp.tokens.numpy(),
                             None if inp.uniforms is None else inp.uniforms.numpy(),
                             inp.temperature, inp.mode, want_debug=True)


def check_valid(g, inp):
    n, out, x = g["accepted_len"], g["out_tokens"], inp.tokens.numpy()
    K = inp.K
    assert ((n >= 0) & (n <= K)).all()
    for b in range(inp.B):
        nb = int(n[b])
        assert (out[b, :nb] == x[b, :nb]).all()
        assert 0 <= out[b, nb] < inp.V
        assert (out[b, nb + 1:] == -1).all()


def assert_parity(g, ref, inp, label=""):
    status = int(g["status"][0])
    assert status == ref["status"], (label, status, ref["status"])
    if status:
        return {"flagged": 0, "B": inp.B}
    check_valid(g, inp)
    if inp.mode == W.MODE_GREEDY:
        np.testing.assert_array_equal(g["accepted_len"], ref["accepted_len"], err_msg=label)
        np.testing.assert_array_equal(g["out_tokens"], ref["out_tokens"], err_msg=label)
        return {"flagged": 0, "B": inp.B}
    flagged = ref["flags"] != 0
    bad = (g["accepted_len"] != ref["accepted_len"]) | (g["out_tokens"] != ref["out_tokens"]).any(1)
    unflagged_bad = np.nonzero(bad & ~flagged)[0]
    if len(unflagged_bad):
        b = int(unflagged_bad[0])
        pytest.fail(f"{label}: {len(unflagged_bad)} unflagged mismatches; first b={b} "
                    f"gpu n={g['accepted_len'][b]} out={g['out_tokens'][b].tolist()} "
                    f"oracle n={ref['accepted_len'][b]} out={ref['out_tokens'][b].tolist()} "
                    f"u={inp.uniforms[b].tolist()} p={ref['p_at'][b].tolist()} "
                    f"q={ref['q_at'][b].tolist()} gpu_flags={g['flags'][b]}")
    tol = 1e-5 if inp.target.dtype == torch.float32 else 2e-3
    if inp.K:
        dp = np.abs(g["p_at"] - ref["p_at"]).max()
        dq = np.abs(g["q_at"] - ref["q_at"]).max()
        assert dp <= tol and dq <= tol, (label, dp, dq)
    print(f"{label}: {inp.B - int(flagged.sum())}/{inp.B} bit-equal, "
          f"{int(flagged.sum())} boundary-flagged ({int((bad & flagged).sum())} of them differ)")
    return {"flagged": int(flagged.sum()), "B": inp.B}


SAMPLE_CASES = [
    # name, B, K, V, dtype, T, recipe
    ("f32_V1000", 16, 4, 1000, torch.float32, 1.0, dict(target_std=3.0, draft_noise=0.5)),
    ("bf16_V7_scalar", 8, 5, 7, torch.bfloat16, 1.0, dict(target_std=2.0, draft_noise=1.0)),
    ("f32_V33_scalar", 8, 3, 33, torch.float32, 0.9, dict(target_std=2.0, draft_noise=1.0)),
    ("f32_V20000_C3", 6, 6, 20000, torch.float32, 0.8, dict(target_std=5.0, independent_draft=True)),
    ("bf16_V70001_C5_scalar", 6, 5, 70001, torch.bfloat16, 1.0,
     dict(target_std=4.0, zipf_s=1.1, draft_noise=1.0)),
    ("bf16_V128256_C8", 4, 5, 128256, torch.bfloat16, 0.7,
     dict(target_std=4.0, zipf_s=1.1, draft_noise=1.0)),
    ("f32_V152064_C8", 3, 16, 152064, torch.float32, 0.8, dict(target_std=5.0, independent_draft=True)),
    ("bf16_V32000_high_accept", 32, 4, 32000, torch.bfloat16, 1.0, dict(target_std=3.0, draft_noise=0.3)),
    ("f32_K0", 6, 0, 5000, torch.float32, 1.0, dict(target_std=3.0)),
    ("f32_Kmax", 3, 64, 300, torch.float32, 1.0, dict(target_std=1.0, draft_noise=0.2)),
    ("f32_V1", 5, 3, 1, torch.float32, 1.0, dict(target_std=1.0)),
    ("f32_V2", 64, 3, 2, torch.float32, 1.0, dict(target_std=1.0, draft_noise=1.0)),
    ("bf16_V3", 64, 2, 3, torch.bfloat16, 1.5, dict(target_std=1.0, draft_noise=1.0)),
    ("bf16_V4096_T0.05", 16, 4, 4096, torch.bfloat16, 0.05, dict(target_std=1.0, draft_noise=0.1)),
    # more sequences than SMs: the fused kernel (the cases above with at most
    # one sequence per SM and short rows take the small-batch kernel)
    ("f32_V1000_B200_fused", 200, 4, 1000, torch.float32, 1.0, dict(target_std=3.0, draft_noise=0.5)),
    ("bf16_V4096_B160_T0.05_fused", 160, 4, 4096, torch.bfloat16, 0.05,
     dict(target_std=1.0, draft_noise=0.1)),
    ("f32_Kmax_B160_fused", 160, 64, 300, torch.float32, 1.0, dict(target_std=1.0, draft_noise=0.2)),
    ("f32_K0_B300_fused", 300, 0, 5000, torch.float32, 1.0, dict(target_std=3.0)),
    # a small batch whose 2K+1 rows just fit the small-batch kernel's 192 KiB
    ("bf16_V10912_K4_smem_limit", 8, 4, 10912, torch.bfloat16, 1.0, dict(target_std=4.0, draft_noise=1.0)),
]


@pytest.mark.parametrize("name,B,K,V,dtype,T,recipe", SAMPLE_CASES, ids=[c[0] for c in SAMPLE_CASES])
def test_sampling_parity(lib, name, B, K, V, dtype, T, recipe):
    inp = W.make_inputs(B, K, V, dtype=dtype, temperature=T, seed=zlib.crc32(name.encode()) % 1000, name=name,
                        **recipe)
    assert_parity(run_gpu(lib, inp), run_oracle(inp), inp, name)


GREEDY_CASES = [
    ("bf16_V32000", 64, 8, 32000, torch.bfloat16, dict(target_std=4.0)),
    ("f32_V1000", 16, 5, 1000, torch.float32, dict(target_std=2.0, greedy_noise=0.5)),
    ("bf16_V7_scalar", 12, 5, 7, torch.bfloat16, dict(target_std=1.0, greedy_noise=0.3)),
    ("f32_V152064", 4, 3, 152064, torch.float32, dict(target_std=5.0, greedy_noise=0.1)),
    ("bf16_K0", 8, 0, 2000, torch.bfloat16, dict(target_std=3.0)),
    ("f32_Kmax", 3, 64, 200, torch.float32, dict(target_std=3.0, greedy_noise=0.01)),
    ("f32_V1", 4, 2, 1, torch.float32, dict()),
    # one CTA per row and K + 1 = 48: the largest sequence whose row count and
    # mismatch bits share one 64-bit word
    ("bf16_K47_one_word", 4, 47, 3000, torch.bfloat16, dict(target_std=3.0, greedy_noise=0.01)),
]


@pytest.mark.parametrize("name,B,K,V,dtype,recipe", GREEDY_CASES, ids=[c[0] for c in GREEDY_CASES])
def test_greedy_parity(lib, name, B, K, V, dtype, recipe):
    inp = W.make_inputs(B, K, V, dtype=dtype, mode=W.MODE_GREEDY, seed=zlib.crc32(name.encode()) % 1000,
                        name=name, **recipe)
    assert_parity(run_gpu(lib, inp), run_oracle(inp), inp, name)


EARLY_EXIT_CASES = [
    # (name, B, K, V, dtype, T, recipe).  One cluster per sequence: low
    # acceptance, moderate, high (every position walked), K = 1, clusters of
    # 1, 2 and 4 CTAs, more clusters than fit at once.  The two-phase schedule
    # (rows too long for a cluster of 8): low acceptance (phase 2 usually
    # skipped) and moderate (it runs).  Short rows go to the small-batch kernel.
    ("ee_f32_independent", 12, 16, 20000, torch.float32, 0.8, dict(target_std=5.0, independent_draft=True)),
    ("ee_bf16_noise", 48, 5, 40000, torch.bfloat16, 1.0, dict(target_std=4.0, zipf_s=1.1, draft_noise=1.0)),
    ("ee_bf16_close", 16, 4, 32000, torch.bfloat16, 1.0, dict(target_std=3.0, draft_noise=0.3)),
    ("ee_f32_K1", 20, 1, 5000, torch.float32, 0.7, dict(target_std=3.0, draft_noise=2.0)),
    ("ee_bf16_K1", 30, 1, 100000, torch.bfloat16, 0.7, dict(target_std=3.0, draft_noise=1.0)),
    ("ee_bf16_c2", 10, 6, 65536, torch.bfloat16, 0.8, dict(target_std=3.0, draft_noise=0.3)),
    ("ee_bf16_c4", 16, 4, 128256, torch.bfloat16, 1.0, dict(target_std=4.0, zipf_s=1.1, draft_noise=1.0)),
    ("ee_bf16_many", 200, 4, 32000, torch.bfloat16, 1.0, dict(target_std=3.0, independent_draft=True)),
    ("ee_bf16_wide", 64, 3, 128256, torch.bfloat16, 1.0, dict(target_std=4.0, zipf_s=1.1, draft_noise=1.0)),
    ("ee_2p_bf16_long_low", 6, 2, 400000, torch.bfloat16, 1.0, dict(target_std=3.0, independent_draft=True)),
    ("ee_2p_bf16_long_mid", 6, 3, 400000, torch.bfloat16, 1.0, dict(target_std=3.0, draft_noise=0.5)),
    ("ee_f32_short", 6, 3, 1000, torch.float32, 1.0, dict(target_std=3.0, independent_draft=True)),
]


def assert_parity_early_exit(g, ref, inp, label):
    """Outputs as in sampling mode; diagnostics for position 0 always, for
    every position when some sequence accepted x_0 (the full pass ran)."""
    assert int(g["status"][0]) == ref["status"] == 0, label
    check_valid(g, inp)
    flagged = ref["flags"] != 0
    bad = (g["accepted_len"] != ref["accepted_len"]) | (g["out_tokens"] != ref["out_tokens"]).any(1)
    assert not (bad & ~flagged).any(), (label, np.nonzero(bad & ~flagged)[0][:5])
    tol = 1e-5 if inp.target.dtype == torch.float32 else 2e-3
    # the diagnostics of positions 0..n, whose rows every schedule reads
    K = g["p_at"].shape[1]
    read = np.arange(K)[None, :] <= ref["accepted_len"][:, None]
    assert np.abs(g["p_at"] - ref["p_at"])[read].max() <= tol, label
    assert np.abs(g["q_at"] - ref["q_at"])[read].max() <= tol, label


@pytest.mark.parametrize("name,B,K,V,dtype,T,recipe", EARLY_EXIT_CASES, ids=[c[0] for c in EARLY_EXIT_CASES])
def test_early_exit_parity(lib, name, B, K, V, dtype, T, recipe):
    inp = W.make_inputs(B, K, V, dtype=dtype, temperature=T, seed=zlib.crc32(name.encode()) % 1000,
                        name=name, **recipe)
    g = run_gpu_mode(lib, inp, "sample_early_exit")
    assert_parity_early_exit(g, run_oracle(inp), inp, name)


def test_early_exit_full_size_long_draft(lib):
    """The fp32 long-draft batch: every sequence rejects its first draft token."""
    inp = W.workload("long_draft_f32_B16_K16_V152064_T0.8")
    g = run_gpu_mode(lib, inp, "sample_early_exit")
    ref = run_oracle(inp)
    assert (ref["accepted_len"] == 0).all()
    assert_parity_early_exit(g, ref, inp, inp.name)


def test_early_exit_workspace_left_zero(lib):
    for name, B, K, V, dtype, T, recipe in EARLY_EXIT_CASES[:3]:
        inp = W.make_inputs(B, K, V, dtype=dtype, temperature=T, seed=7, name=name, **recipe)
        dt = lib.DTYPE_BF16 if dtype == torch.bfloat16 else lib.DTYPE_F32
        ws = torch.zeros(lib.workspace_size(B, K, V, dt, lib.MODE_SAMPLE_EARLY_EXIT),
                         dtype=torch.uint8, device="cuda")
        for _ in range(2):
            lib.verify(_dev(inp.target), _dev(inp.draft), _dev(inp.tokens), _dev(inp.uniforms),
                       T, "sample_early_exit", workspace=ws)
        torch.cuda.synchronize()
        assert int(ws.count_nonzero().item()) == 0, name


def test_greedy_ties_take_the_lowest_index(lib):
    """Integer-valued bf16 logits: most rows have tied maxima, some across
    the split of a row into segments."""
    g = torch.Generator().manual_seed(5)
    B, K, V = 32, 6, 40000
    t = torch.randint(0, 3, (B, K + 1, V), generator=g).to(torch.bfloat16)
    t[:, :, -1] = 2.0          # a tie at the very end of every row
    t[0, :, :] = 0.0           # fully tied rows
    t[1, :, :] = float("-inf")
    x = t[:, :K].float().argmax(-1).to(torch.int32)
    x[::3, 2] = 7              # some mismatches
    inp = W.Inputs("ties", W.MODE_GREEDY, B, K, V, 1.0, t.contiguous(), None, x.contiguous(), None)
    assert_parity(run_gpu(lib, inp), run_oracle(inp), inp, "ties")


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_full_size_workloads(lib, name):
    inp = W.workload(name)
    assert_parity(run_gpu(lib, inp), run_oracle(inp), inp, name)


def test_maximum_vocabulary(lib):
    V = lib.MAX_V
    inp = W.make_inputs(1, 1, V, dtype=torch.float32, temperature=1.0, target_std=3.0,
                        draft_noise=1.0, seed=4, name="maxV")
    assert_parity(run_gpu(lib, inp), run_oracle(inp), inp, "maxV")


def test_identical_models_accept_everything(lib):
    inp = W.make_inputs(16, 5, 3000, dtype=torch.bfloat16, seed=9, name="same")
    inp.draft = inp.target[:, :5].clone()
    inp.tokens = torch.randint(0, 3000, (16, 5), dtype=torch.int32)
    g, ref = run_gpu(lib, inp), run_oracle(inp)
    assert (g["accepted_len"] == 5).all()
    assert_parity(g, ref, inp, "same")


def test_neg_inf_logits_are_allowed(lib):
    inp = W.make_inputs(8, 4, 2000, dtype=torch.float32, seed=10, name="neginf")
    inp.target[:, :, ::3] = float("-inf")
    inp.draft[:, :, 1::3] = float("-inf")
    g, ref = run_gpu(lib, inp), run_oracle(inp)
    assert int(g["status"][0]) == 0
    assert_parity(g, ref, inp, "neginf")
    zero = inp.target.numpy()[np.arange(8)[:, None], np.arange(5)[None], g["out_tokens"].clip(0)]
    emitted = g["out_tokens"] >= 0
    assert np.isfinite(zero[emitted]).all()  # never emits a token the target gives no mass


@pytest.mark.parametrize("what", ["token", "nan", "posinf", "uniform", "allneginf"])
def test_data_errors_set_status_and_stay_in_range(lib, what):
    inp = W.make_inputs(6, 3, 4000, dtype=torch.float32, seed=11, name=what)
    if what == "token":
        inp.tokens[2, 1] = 4000
    elif what == "nan":
        inp.target[3, 2, 17] = float("nan")
    elif what == "posinf":
        inp.draft[1, 0, 5] = float("inf")
    elif what == "uniform":
        inp.uniforms[4, 3] = 1.0
    else:
        inp.target[0, 1, :] = float("-inf")
    g, ref = run_gpu(lib, inp), run_oracle(inp)
    assert int(g["status"][0]) == ref["status"] != 0
    assert ((g["accepted_len"] >= 0) & (g["accepted_len"] <= 3)).all()
    assert ((g["out_tokens"] >= -1) & (g["out_tokens"] < 4000)).all()
    # sequences without a data error are unaffected
    good = ref["accepted_len"] >= 0
    ok = good & (ref["flags"] == 0)
    np.testing.assert_array_equal(g["accepted_len"][ok], ref["accepted_len"][ok])
    np.testing.assert_array_equal(g["out_tokens"][ok], ref["out_tokens"][ok])


@pytest.mark.parametrize("what", ["token", "nan", "posinf", "uniform", "neginf_row"])
def test_early_exit_cluster_data_errors(lib, what):
    """Data errors at position 0 (whose rows every schedule reads) on the
    early-exit kernel whose clusters walk the positions: the same status as
    the oracle, outputs in range, the other sequences unaffected."""
    inp = W.make_inputs(6, 3, 40000, dtype=torch.float32, seed=13, name=what, target_std=3.0,
                        independent_draft=True)
    if what == "token":
        inp.tokens[2, 0] = 40000
    elif what == "nan":
        inp.target[3, 0, 17] = float("nan")
    elif what == "posinf":
        inp.draft[1, 0, 5] = float("inf")
    elif what == "uniform":
        inp.uniforms[4, 0] = 1.0
    else:
        inp.target[0, 0, :] = float("-inf")
    g, ref = run_gpu_mode(lib, inp, "sample_early_exit"), run_oracle(inp)
    assert int(g["status"][0]) == ref["status"] != 0, what
    assert ((g["accepted_len"] >= 0) & (g["accepted_len"] <= 3)).all()
    assert ((g["out_tokens"] >= -1) & (g["out_tokens"] < 40000)).all()
    good = ref["accepted_len"] >= 0
    ok = good & (ref["flags"] == 0)
    np.testing.assert_array_equal(g["accepted_len"][ok], ref["accepted_len"][ok])
    np.testing.assert_array_equal(g["out_tokens"][ok], ref["out_tokens"][ok])


def test_greedy_data_errors(lib):
    inp = W.make_inputs(5, 3, 3000, dtype=torch.bfloat16, mode=W.MODE_GREEDY, seed=12)
    inp.target[1, 2, 100] = float("nan")
    inp.tokens[3, 0] = -5
    g, ref = run_gpu(lib, inp), run_oracle(inp)
    assert int(g["status"][0]) == ref["status"] == 3


@pytest.mark.parametrize("shape", [(300, 4, 1000, torch.float32), (8, 4, 3000, torch.bfloat16),
                                   (64, 8, 32000, torch.bfloat16)],
                         ids=["fused", "small_batch", "greedy"])
def test_bit_identical_over_100_runs(lib, shape):
    """Races in the reductions or the arrival protocol would make repeated runs
    on the same inputs differ: 100 runs must give identical outputs,
    diagnostics included."""
    B, K, V, dtype = shape
    mode = W.MODE_GREEDY if V == 32000 else W.MODE_SAMPLE
    inp = W.make_inputs(B, K, V, dtype=dtype, mode=mode, temperature=0.9, target_std=4.0,
                        draft_noise=1.0, seed=17)
    first = run_gpu(lib, inp)
    for _ in range(99):
        cur = run_gpu(lib, inp)
        for k in first:
            assert np.array_equal(cur[k], first[k]), k


def test_deterministic_and_workspace_left_zero(lib):
    inp = W.make_inputs(64, 5, 50000, dtype=torch.bfloat16, temperature=0.9, target_std=4.0,
                        draft_noise=1.0, seed=13)
    dev = [_dev(t) for t in (inp.target, inp.draft, inp.tokens, inp.uniforms)]
    nbytes = lib.workspace_size(64, 5, 50000, lib.DTYPE_BF16, lib.MODE_SAMPLE)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    first = None
    for _ in range(100):
        acc, out = lib.verify(*dev, inp.temperature, "sample", workspace=ws)
        torch.cuda.synchronize()
        cur = (acc.cpu().numpy(), out.cpu().numpy())
        if first is None:
            first = cur
        assert np.array_equal(cur[0], first[0]) and np.array_equal(cur[1], first[1])
    # the whole workspace (counters, masks, candidates) is back to zero
    assert int(ws.count_nonzero().item()) == 0
    g = W.make_inputs(64, 8, 32000, dtype=torch.bfloat16, mode=W.MODE_GREEDY, seed=14)
    wsg = torch.zeros(lib.workspace_size(64, 8, 32000, 1, 1), dtype=torch.uint8, device="cuda")
    lib.verify(_dev(g.target), None, _dev(g.tokens), None, 1.0, "greedy", workspace=wsg)
    torch.cuda.synchronize()
    assert int(wsg.count_nonzero().item()) == 0


def test_greedy_ignores_draft_uniforms_and_temperature(lib):
    inp = W.make_inputs(4, 3, 1000, dtype=torch.float32, mode=W.MODE_GREEDY, seed=15)
    acc, out = lib.verify(_dev(inp.target), None, _dev(inp.tokens), None, float("nan"), "greedy")
    ref = run_oracle(inp)
    np.testing.assert_array_equal(out.cpu().numpy(), ref["out_tokens"])


def test_host_tensors_roundtrip_through_the_device(lib):
    inp = W.make_inputs(8, 4, 3000, dtype=torch.float32, seed=16)
    acc, out = lib.verify(inp.target.pin_memory(), inp.draft.pin_memory(),
                          inp.tokens.pin_memory(), inp.uniforms.pin_memory(), 1.0, "sample")
    assert not acc.is_cuda
    ref = run_oracle(inp)
    ok = ref["flags"] == 0
    np.testing.assert_array_equal(out.numpy()[ok], ref["out_tokens"][ok])


def test_bad_arguments_raise_before_launch(lib):
    t = torch.zeros((2, 3, 10), device="cuda")
    with pytest.raises(TypeError):
        lib.verify(t, torch.zeros((2, 2, 10), device="cuda"), torch.zeros((2, 2), dtype=torch.int64,
                   device="cuda"), torch.zeros((2, 3), device="cuda"), 1.0)
    with pytest.raises(lib.SpecVerifyError):
        lib.verify(t, torch.zeros((2, 2, 10), device="cuda"),
                   torch.zeros((2, 2), dtype=torch.int32, device="cuda"),
                   torch.zeros((2, 3), device="cuda"), 0.0)


DRAFT_SAMPLE_CASES = [
    # (name, rows shape, V, dtype, T): clusters of 1, 2, 4 and 8 CTAs per
    # row, short and ragged warp ranges, more rows than resident CTAs, a cold
    # temperature, and rows too long for a cluster (the K = 0 verify)
    ("ds_f32_short", (5, 3), 1000, torch.float32, 1.0),
    ("ds_f32_tiny", (7,), 36, torch.float32, 1.0),
    ("ds_bf16_32000", (8, 4), 32000, torch.bfloat16, 1.0),
    ("ds_bf16_65536_c2", (12,), 65536, torch.bfloat16, 0.9),
    ("ds_bf16_128256", (40,), 128256, torch.bfloat16, 0.7),
    ("ds_f32_152064", (16,), 152064, torch.float32, 0.8),
    ("ds_bf16_32000_many", (4, 300), 32000, torch.bfloat16, 1.0),
    ("ds_bf16_32768_limit", (310,), 32768, torch.bfloat16, 0.7),
    ("ds_f32_16384_limit", (161,), 16384, torch.float32, 1.3),
    ("ds_bf16_4096_T0.05", (700,), 4096, torch.bfloat16, 0.05),
    ("ds_bf16_393216_c8", (3,), 393216, torch.bfloat16, 1.0),
    ("ds_bf16_100008_c4_ragged", (6,), 100008, torch.bfloat16, 1.1),
    ("ds_f32_24580_c2_ragged", (9,), 24580, torch.float32, 0.9),
    ("ds_bf16_400000_verify", (3,), 400000, torch.bfloat16, 1.0),
]


@pytest.mark.parametrize("name,shape,V,dtype,T", DRAFT_SAMPLE_CASES, ids=[c[0] for c in DRAFT_SAMPLE_CASES])
def test_draft_sample_parity(lib, name, shape, V, dtype, T):
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()) % 1000)
    x = (torch.randn(*shape, V, generator=g) * 4.0).to(dtype)
    x[..., ::11] = float("-inf")
    u = torch.rand(*shape, generator=g)
    ref = oracle.draft_sample_ref(W.as_numpy_logits(x), u.numpy(), T)
    ws_bytes = lib.workspace_size(int(np.prod(shape)), 0, V,
                                  lib.DTYPE_BF16 if dtype == torch.bfloat16 else lib.DTYPE_F32,
                                  lib.MODE_SAMPLE)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    tok, q, status = lib.draft_sample(_dev(x), _dev(u), T, workspace=ws, debug=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    tok, q = tok.cpu().numpy(), q.cpu().numpy()
    flagged = ref["flags"] != 0
    assert not ((tok != ref["tokens"]) & ~flagged).any(), (name, int(((tok != ref["tokens"]) & ~flagged).sum()))
    tol = 1e-5 if dtype == torch.float32 else 2e-3
    assert np.abs(q - ref["q_at"]).max() <= tol, name
    assert int(ws.count_nonzero().item()) == 0  # left zero-filled


def test_draft_sample_nonfinite_rows(lib):
    """A row with a NaN, one with +inf and one with no finite logit set
    SPEC_DATA_NONFINITE_LOGIT; the finite rows still equal the oracle."""
    g = torch.Generator().manual_seed(77)
    for V, dtype in ((32000, torch.bfloat16), (152064, torch.float32)):
        x = (torch.randn(6, V, generator=g) * 3.0).to(dtype)
        x[1, 17] = float("nan")
        x[2, V - 3] = float("inf")
        x[3, :] = float("-inf")
        u = torch.rand(6, generator=g)
        tok, q, status = lib.draft_sample(_dev(x), _dev(u), 1.0, debug=True)
        torch.cuda.synchronize()
        assert int(status.item()) & lib.DATA_NONFINITE_LOGIT
        fine = [0, 4, 5]
        ref = oracle.draft_sample_ref(W.as_numpy_logits(x[fine]), u[fine].numpy(), 1.0)
        ok = ref["flags"] == 0
        np.testing.assert_array_equal(tok.cpu().numpy()[fine][ok], ref["tokens"][ok])
        assert ((tok.cpu().numpy() >= 0) & (tok.cpu().numpy() < V)).all()


def test_draft_sample_rejects_unaligned_rows(lib):
    x = torch.randn(4, 1001, device="cuda")  # 4004-byte rows: not 16-byte multiples
    u = torch.rand(4, device="cuda")
    with pytest.raises(lib.SpecVerifyError):
        lib.draft_sample(x, u, 1.0)


# --------------------------------------------------------------------------
# Speculative Rejection's cut: r_cut, the kept count and the kept indices are
# bit-equal to the oracle's (r_cut is one fixed double expression of two
# order statistics, and the keep test is exact).
# --------------------------------------------------------------------------
CUT_CASES = [
    # (name, G, N, alpha, score kind): warp kernel (N <= 1024, four register
    # widths, ragged G and N), block kernel (N > 1024), ties, alpha edges
    ("cut_n1", 3, 1, 0.5, "normal"),
    ("cut_n5", 17, 5, 0.6, "normal"),
    ("cut_n100", 33, 100, 0.25, "normal"),
    ("cut_n200_ties", 40, 200, 0.5, "ties"),
    ("cut_n513", 9, 513, 0.9, "normal"),
    ("cut_n1000", 1001, 1000, 0.5, "normal"),
    ("cut_n1000_a0", 50, 1000, 0.0, "normal"),
    ("cut_n1000_a1", 50, 1000, 1.0, "normal"),
    ("cut_n1000_tiny_g", 64, 1000, 1e-300, "ties"),
    ("cut_n1024_ties", 16, 1024, 0.731, "ties"),
    ("cut_n1025", 7, 1025, 0.5, "normal"),
    ("cut_n5000_ties", 5, 5000, 0.3, "ties"),
    ("cut_n70000", 2, 70000, 0.77, "normal"),
]


def _assert_cut_equal(got, ref, name):
    r, n, acc = (t.cpu().numpy() for t in got)
    np.testing.assert_array_equal(np.isnan(r), np.isnan(ref["r_cut"]), err_msg=name)
    ok = ~np.isnan(r)
    assert np.array_equal(r[ok], ref["r_cut"][ok]), (name, np.flatnonzero(r[ok] != ref["r_cut"][ok])[:5])
    np.testing.assert_array_equal(n, ref["n_accepted"], err_msg=name)
    np.testing.assert_array_equal(acc, ref["accepted"], err_msg=name)


@pytest.mark.parametrize("name,G,N,alpha,kind", CUT_CASES, ids=[c[0] for c in CUT_CASES])
def test_rejection_cut_parity(lib, name, G, N, alpha, kind):
    s = W.make_scores(G, N, kind=kind, seed=zlib.crc32(name.encode()) % 1000)
    ref = oracle.rejection_cut_ref(s.numpy(), alpha)
    got = lib.rejection_cut(_dev(s), alpha, debug=True)
    torch.cuda.synchronize()
    assert int(got[3].item()) == 0
    _assert_cut_equal(got[:3], ref, name)


@pytest.mark.parametrize("N", [100, 1000, 2000])
def test_rejection_cut_extreme_scores(lib, N):
    """Scores at the ends of the fp32 range (keys next to the padding of a
    ragged row), all-equal rows and tiny spreads."""
    s = W.make_scores(24, N, seed=N + 1)
    s[0] = -3.0e38
    s[1, : N // 2] = -3.0e38
    s[2, ::3] = 3.0e38
    s[3] = 1e-40  # subnormal, all equal
    s[4] = s[4] * 1e-30
    s[5, ::2] = -0.0
    s[5, 1::2] = 0.0
    for alpha in (0.0, 0.37, 1.0):
        ref = oracle.rejection_cut_ref(s.numpy(), alpha)
        got = lib.rejection_cut(_dev(s), alpha)
        torch.cuda.synchronize()
        _assert_cut_equal(got, ref, f"extreme N={N} alpha={alpha}")


def test_rejection_cut_full_size(lib):
    """The benchmarked workload (16384 prompts of 1000 scores), every output."""
    spec = W.REJECTION_WORKLOADS["rejection_cut_f32_G16384_N1000_a0.5"]
    s = W.make_scores(spec["G"], spec["N"], kind=spec["kind"], seed=0)
    ref = oracle.rejection_cut_ref(s.numpy(), spec["alpha"])
    got = lib.rejection_cut(_dev(s), spec["alpha"])
    torch.cuda.synchronize()
    _assert_cut_equal(got, ref, "full")


@pytest.mark.parametrize("N", [300, 3000])
def test_rejection_cut_nonfinite_scores(lib, N):
    s = W.make_scores(12, N, seed=N)
    s[2, 7] = float("nan")
    s[5, N - 1] = float("inf")
    s[9, 0] = float("-inf")
    ref = oracle.rejection_cut_ref(s.numpy(), 0.4)
    got = lib.rejection_cut(_dev(s), 0.4, debug=True)
    torch.cuda.synchronize()
    assert ref["status"] == oracle.DATA_SCORE  # the two sides number their bits on their own
    assert int(got[3].item()) == lib.DATA_NONFINITE_SCORE
    _assert_cut_equal(got[:3], ref, f"nonfinite N={N}")


def test_rejection_cut_empty_batch(lib):
    r, n, acc = lib.rejection_cut(torch.zeros((0, 10), device="cuda"), 0.5)
    torch.cuda.synchronize()
    assert r.numel() == 0 and n.numel() == 0 and acc.numel() == 0


# --------------------------------------------------------------------------
# Speculative contrastive decoding: the same bar as sampling mode, with the
# oracle's contrastive target (the temperature passed to both sides as the
# same fp32 value, so the head's threshold is the same double).
# --------------------------------------------------------------------------
SCD_CASES = [
    # name, B, K, V, dtype, T, alpha, recipe  (cluster sizes 1, 2, 8 at two and one CTA per SM)
    ("scd_f32_V1000", 16, 4, 1000, torch.float32, 1.0, 0.1, dict(target_std=3.0, amateur_noise=1.0)),
    ("scd_bf16_V32000", 16, 4, 32000, torch.bfloat16, 0.7, 0.1, dict(target_std=3.0, amateur_noise=0.5)),
    ("scd_bf16_V128256", 6, 5, 128256, torch.bfloat16, 1.0, 0.1,
     dict(target_std=4.0, zipf_s=1.1, amateur_noise=1.0)),
    ("scd_f32_V152064_low_accept", 3, 8, 152064, torch.float32, 0.8, 0.05,
     dict(target_std=5.0, independent_amateur=True)),
    ("scd_f32_alpha0", 8, 3, 5000, torch.float32, 1.0, 0.0, dict(target_std=3.0, amateur_noise=1.0)),
    ("scd_f32_K0", 6, 0, 4096, torch.float32, 1.0, 0.2, dict(target_std=3.0)),
    ("scd_bf16_V1024_T0.05", 16, 3, 1024, torch.bfloat16, 0.05, 0.3, dict(target_std=1.0, amateur_noise=0.1)),
    # heads too wide to remember vector by vector: the slice is read again
    ("scd_f32_V152064_alpha0_rescan", 2, 3, 152064, torch.float32, 1.0, 0.0,
     dict(target_std=3.0, amateur_noise=1.0)),
    ("scd_f32_V152064_flat_rescan", 2, 3, 152064, torch.float32, 1.0, 0.01,
     dict(target_std=0.5, amateur_noise=0.3)),
]


def run_scd(lib, inp, alpha, T32):
    res = lib.verify_scd(_dev(inp.target), _dev(inp.draft), _dev(inp.tokens), _dev(inp.uniforms),
                         T32, alpha, debug=True)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in res.items()}


def scd_oracle(inp, alpha, T32):
    return oracle.scd_verify_ref(W.as_numpy_logits(inp.target), W.as_numpy_logits(inp.draft),
                                 inp.tokens.numpy(), inp.uniforms.numpy(), T32, alpha,
                                 want_debug=True)


@pytest.mark.parametrize("name,B,K,V,dtype,T,alpha,recipe", SCD_CASES, ids=[c[0] for c in SCD_CASES])
def test_scd_parity(lib, name, B, K, V, dtype, T, alpha, recipe):
    inp = W.make_scd_inputs(B, K, V, dtype=dtype, temperature=T, name=name,
                            seed=zlib.crc32(name.encode()) % 1000, **recipe)
    T32 = float(np.float32(T))
    assert_parity(run_scd(lib, inp, alpha, T32), scd_oracle(inp, alpha, T32), inp, name)


def test_scd_full_size(lib):
    """The benchmarked workload (64 sequences, K = 5, V = 128256 bf16)."""
    spec = dict(W.SCD_WORKLOADS["scd_bf16_B64_K5_V128256_T1.0_a0.1"])
    alpha = spec.pop("alpha")
    inp = W.make_scd_inputs(seed=0, **spec)
    T32 = float(np.float32(inp.temperature))
    assert_parity(run_scd(lib, inp, alpha, T32), scd_oracle(inp, alpha, T32), inp, "scd full")


def test_scd_tightest_head_is_greedy_on_gpu(lib):
    inp = W.make_scd_inputs(32, 5, 32000, dtype=torch.bfloat16, target_std=4.0, amateur_noise=2.0,
                            seed=9)
    g = run_scd(lib, inp, 1.0, 1.0)
    ref = oracle.verify_ref(W.as_numpy_logits(inp.target), None, inp.tokens.numpy(), None,
                            mode=oracle.MODE_GREEDY)
    np.testing.assert_array_equal(g["accepted_len"], ref["accepted_len"])
    np.testing.assert_array_equal(g["out_tokens"], ref["out_tokens"])


def test_scd_data_errors_and_workspace(lib):
    inp = W.make_scd_inputs(6, 3, 2048, dtype=torch.float32, target_std=3.0, seed=12)
    inp.draft[1, 2, 100] = float("nan")
    top = int(inp.target[3, 1].argmax())
    inp.draft[3, 1, top] = float("-inf")  # an unbounded contrast in the head
    B, K, V = inp.B, inp.K, inp.V
    ws = torch.zeros(lib.workspace_size(B, K, V, lib.DTYPE_F32, lib.MODE_SAMPLE), dtype=torch.uint8,
                     device="cuda")
    g = lib.verify_scd(_dev(inp.target), _dev(inp.draft), _dev(inp.tokens), _dev(inp.uniforms), 1.0,
                       0.1, workspace=ws, debug=True)
    torch.cuda.synchronize()
    ref = oracle.scd_verify_ref(inp.target.numpy(), inp.draft.numpy(), inp.tokens.numpy(),
                                inp.uniforms.numpy(), 1.0, 0.1, want_debug=True)
    assert ref["status"] == oracle.DATA_LOGIT
    assert int(g["status"].item()) == lib.DATA_NONFINITE_LOGIT
    ok = (ref["accepted_len"] >= 0) & (ref["flags"] == 0)
    assert ok.sum() >= 3
    np.testing.assert_array_equal(g["accepted_len"].cpu().numpy()[ok], ref["accepted_len"][ok])
    assert int(ws.count_nonzero().item()) == 0  # left zero-filled


@pytest.mark.parametrize("N", [2, 31, 32, 33, 128, 129, 256, 257, 512, 1023, 1024, 2048, 4097])
def test_rejection_cut_register_width_edges(lib, N):
    """Row lengths at and around each register width of the warp kernel
    (4, 8, 16, 32 scores a lane) and the switch to one CTA per prompt."""
    s = W.make_scores(5, N, seed=N + 7)
    for alpha in (0.0, 0.5, 0.999, 1.0):
        ref = oracle.rejection_cut_ref(s.numpy(), alpha)
        got = lib.rejection_cut(_dev(s), alpha)
        torch.cuda.synchronize()
        _assert_cut_equal(got, ref, f"N={N} alpha={alpha}")


def test_rejection_cut_one_prompt_one_score(lib):
    s = torch.tensor([[-2.5]])
    r, n, acc = lib.rejection_cut(_dev(s), 0.3)
    torch.cuda.synchronize()
    assert r.item() == -2.5 and n.item() == 1 and acc.tolist() == [[0]]


SCD_EDGE_CASES = [
    # name, B, K, V, dtype, T, alpha: the largest K, a tiny vocabulary, one draft position
    ("scd_f32_Kmax", 3, 64, 256, torch.float32, 1.0, 0.2),
    ("scd_f32_V4", 64, 2, 4, torch.float32, 1.0, 0.5),
    ("scd_bf16_V8", 64, 3, 8, torch.bfloat16, 0.8, 0.1),
    ("scd_bf16_K1", 32, 1, 32000, torch.bfloat16, 1.0, 0.1),
]


@pytest.mark.parametrize("name,B,K,V,dtype,T,alpha", SCD_EDGE_CASES, ids=[c[0] for c in SCD_EDGE_CASES])
def test_scd_edge_shapes(lib, name, B, K, V, dtype, T, alpha):
    inp = W.make_scd_inputs(B, K, V, dtype=dtype, temperature=T, name=name, target_std=2.0,
                            amateur_noise=0.5, seed=zlib.crc32(name.encode()) % 1000)
    T32 = float(np.float32(T))
    assert_parity(run_scd(lib, inp, alpha, T32), scd_oracle(inp, alpha, T32), inp, name)


def test_scd_empty_batch(lib):
    t = torch.zeros((0, 3, 1024), device="cuda")
    n, out = lib.verify_scd(t, t.clone(), torch.zeros((0, 2), dtype=torch.int32, device="cuda"),
                            torch.zeros((0, 3), device="cuda"), 1.0, 0.1)
    torch.cuda.synchronize()
    assert n.numel() == 0 and out.numel() == 0
