"""CPU-only checks of the C-ABI library: it loads, exports every symbol the
header declares, sizes its workspace, and rejects bad arguments on the host
before any CUDA call.  No kernel is launched here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def binding():
    import __graft_entry__
    __graft_entry__.build()
    from draft_verify_acceptance_gb300 import binding
    return binding


def _declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"SPEC_API\s+[\w\s\*]+?\b(spec_\w+)\s*\(", src)))


def _header_defines():
    src = open(HEADER).read()
    out = {}
    for name, val in re.findall(r"#define\s+(SPEC_\w+)\s+\(?([0-9x]+(?:\s*<<\s*\d+)?)\)?", src):
        out[name] = eval(val)
    for name, val in re.findall(r"(SPEC_\w+)\s*=\s*(\d+)", src):
        out[name] = int(val)
    return out


def test_library_exports_every_declared_symbol(binding):
    names = _declared_functions()
    assert set(names) == {"spec_verify", "spec_verify_ex", "spec_verify_workspace_size",
                          "spec_status_string", "spec_verify_static", "spec_draft_sample",
                          "spec_rejection_cut", "spec_verify_scd", "spec_set_wait_limit"}
    assert set(names) == set(binding.EXPORTS)
    lib = ctypes.CDLL(binding.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    dyn = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH],
                         capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in dyn.splitlines() if " T " in line}
    assert set(names) <= exported
    # nothing of the implementation leaks out of the C ABI
    assert not [s for s in exported if "specv" in s]


def test_header_constants_match_binding(binding):
    d = _header_defines()
    assert d["SPEC_OK"] == binding.OK
    assert d["SPEC_ERR_INVALID_ARG"] == binding.ERR_INVALID_ARG
    assert d["SPEC_ERR_UNSUPPORTED"] == binding.ERR_UNSUPPORTED
    assert d["SPEC_ERR_CUDA"] == binding.ERR_CUDA
    assert d["SPEC_ERR_SCRATCH_LIMIT"] == binding.ERR_SCRATCH_LIMIT
    assert d["SPEC_STATIC_SCRATCH_BYTES"] == binding.STATIC_SCRATCH_BYTES
    assert d["SPEC_MODE_SAMPLE"] == binding.MODE_SAMPLE
    assert d["SPEC_MODE_GREEDY"] == binding.MODE_GREEDY
    assert d["SPEC_MODE_SAMPLE_EARLY_EXIT"] == binding.MODE_SAMPLE_EARLY_EXIT
    assert d["SPEC_DTYPE_F32"] == binding.DTYPE_F32
    assert d["SPEC_DTYPE_BF16"] == binding.DTYPE_BF16
    assert d["SPEC_MAX_K"] == binding.MAX_K
    assert d["SPEC_MAX_V"] == binding.MAX_V
    assert d["SPEC_DATA_TOKEN_RANGE"] == binding.DATA_TOKEN_RANGE
    assert d["SPEC_DATA_NONFINITE_LOGIT"] == binding.DATA_NONFINITE_LOGIT
    assert d["SPEC_DATA_UNIFORM_RANGE"] == binding.DATA_UNIFORM_RANGE
    assert d["SPEC_DEVICE_WAIT_TIMEOUT"] == binding.DEVICE_WAIT_TIMEOUT
    assert d["SPEC_FLAG_RATIO"] == binding.FLAG_RATIO
    assert d["SPEC_FLAG_CDF"] == binding.FLAG_CDF


def test_data_error_bits_agree_with_the_oracle():
    import oracle
    from draft_verify_acceptance_gb300 import binding
    assert oracle.DATA_TOKEN == binding.DATA_TOKEN_RANGE
    assert oracle.DATA_LOGIT == binding.DATA_NONFINITE_LOGIT
    assert oracle.DATA_UNIFORM == binding.DATA_UNIFORM_RANGE


def test_workspace_size(binding):
    ws = binding.workspace_size
    assert ws(64, 8, 32000, binding.DTYPE_BF16, binding.MODE_GREEDY) % 256 == 0
    assert ws(64, 8, 32000, 1, 1) >= 64 * 32 + 64 * 9 * 8
    assert ws(0, 4, 10, 0, 0) == 0 or ws(0, 4, 10, 0, 0) % 256 == 0
    assert ws(-1, 4, 10, 0, 0) == 0
    assert ws(4, 65, 10, 0, 0) == 0
    assert ws(4, 4, 0, 0, 0) == 0
    assert ws(4, 4, 10, 2, 0) == 0
    assert ws(4, 4, 10, 0, 3) == 0
    assert ws(4, 4, 10, 0, binding.MODE_SAMPLE_EARLY_EXIT) == ws(4, 4, 10, 0, binding.MODE_SAMPLE)
    assert ws(4, 4, binding.MAX_V + 1, 0, 0) == 0


def _raw_call(binding, **kw):
    """spec_verify_ex with fake (never dereferenced) aligned pointers.  The
    default workspace size is too small, so even a call whose other arguments
    are all valid stops at the host-side checks and never reaches a launch."""
    fake = ctypes.c_void_p(1 << 20)
    args = dict(target=fake, draft=fake, tokens=fake, uniforms=fake, B=2, K=3, V=100, dtype=0,
                T=1.0, mode=0, acc=fake, out=fake, ws=fake, ws_bytes=16, stream=None,
                p=None, q=None, flags=None, status=None)
    args.update(kw)
    return binding._lib.spec_verify_ex(
        args["target"], args["draft"], args["tokens"], args["uniforms"], args["B"], args["K"],
        args["V"], args["dtype"], args["T"], args["mode"], args["acc"], args["out"], args["ws"],
        args["ws_bytes"], args["stream"], args["p"], args["q"], args["flags"], args["status"])


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), 1), (dict(K=-1), 1), (dict(V=0), 1), (dict(dtype=7), 1), (dict(mode=3), 1),
    (dict(K=65), 2), (dict(V=(1 << 22) + 1), 2),
    (dict(T=0.0), 1), (dict(T=-1.0), 1), (dict(T=float("inf")), 1), (dict(T=float("nan")), 1),
    (dict(target=None), 1), (dict(tokens=None), 1), (dict(acc=None), 1), (dict(out=None), 1),
    (dict(draft=None), 1), (dict(uniforms=None), 1),
    (dict(ws=None, ws_bytes=1 << 20), 1), (dict(ws_bytes=16), 1),
    (dict(ws=ctypes.c_void_p((1 << 20) + 8), ws_bytes=1 << 20), 1),
    (dict(target=ctypes.c_void_p((1 << 20) + 2)), 1),
    (dict(tokens=ctypes.c_void_p((1 << 20) + 2)), 1),
])
def test_invalid_arguments_rejected_on_host(binding, kw, code):
    assert _raw_call(binding, **kw) == code


def test_greedy_needs_neither_draft_nor_uniforms_nor_temperature(binding):
    import torch
    if torch.cuda.is_available():
        pytest.skip("would launch on fake pointers; the GPU suite covers this with real tensors")
    # argument checks pass; with no GPU the call then fails at the CUDA layer
    rc = _raw_call(binding, mode=1, draft=None, uniforms=None, T=float("nan"), ws_bytes=1 << 20)
    assert rc == binding.ERR_CUDA


def test_empty_batch_is_a_noop(binding):
    assert _raw_call(binding, B=0, target=None, acc=None, out=None, ws=None) == 0


def test_status_strings(binding):
    assert binding.status_string(0) == "ok"
    assert "invalid" in binding.status_string(1)
    assert binding.status_string(99) == "unknown status"


def test_python_binding_refuses_cpu_fallback(binding):
    import torch
    t = torch.zeros((2, 3, 10))
    with pytest.raises(Exception):
        binding._call(t, None, None, None, 1.0, "greedy", False, None, None)


def test_draft_sample_host_checks(binding):
    """spec_draft_sample's argument errors return before any launch (fake,
    never dereferenced pointers)."""
    f = binding._lib.spec_draft_sample
    P, fake = ctypes.c_void_p, ctypes.c_void_p(1 << 20)
    ws = binding.workspace_size(4, 0, 1024, binding.DTYPE_F32, binding.MODE_SAMPLE)
    def call(R=4, V=1024, dtype=binding.DTYPE_F32, T=1.0, logits=fake, u=fake, tok=fake, nbytes=ws):
        return f(logits, u, R, V, dtype, T, tok, None, fake, nbytes, None, None)
    assert call(R=-1) == binding.ERR_INVALID_ARG
    assert call(V=0) == binding.ERR_INVALID_ARG
    assert call(dtype=7) == binding.ERR_INVALID_ARG
    assert call(T=0.0) == binding.ERR_INVALID_ARG
    assert call(T=float("nan")) == binding.ERR_INVALID_ARG
    assert call(logits=None) == binding.ERR_INVALID_ARG
    assert call(u=None) == binding.ERR_INVALID_ARG
    assert call(tok=None) == binding.ERR_INVALID_ARG
    assert call(nbytes=16) == binding.ERR_INVALID_ARG
    assert call(V=binding.MAX_V + 1) == binding.ERR_UNSUPPORTED
    wsu = binding.workspace_size(4, 0, 1001, binding.DTYPE_F32, binding.MODE_SAMPLE)
    assert call(V=1001, nbytes=wsu) == binding.ERR_UNSUPPORTED  # rows not 16-byte multiples
    assert call(R=0) == binding.OK


def test_rejection_cut_host_checks(binding):
    """spec_rejection_cut's argument errors return before any launch (fake,
    never dereferenced pointers); G == 0 is a no-op."""
    f = binding._lib.spec_rejection_cut
    fake = ctypes.c_void_p(1 << 20)
    def call(G=4, N=1000, alpha=0.5, s=fake, r=fake, n=fake, acc=fake, st=None):
        return f(s, G, N, alpha, r, n, acc, None, st)
    assert binding.DATA_NONFINITE_SCORE == _header_defines()["SPEC_DATA_NONFINITE_SCORE"]
    assert call(G=-1) == binding.ERR_INVALID_ARG
    assert call(N=0) == binding.ERR_INVALID_ARG
    assert call(N=-3) == binding.ERR_INVALID_ARG
    for a in (-0.01, 1.01, float("nan"), float("inf")):
        assert call(alpha=a) == binding.ERR_INVALID_ARG
    assert call(s=None) == binding.ERR_INVALID_ARG
    assert call(r=None) == binding.ERR_INVALID_ARG
    assert call(n=None) == binding.ERR_INVALID_ARG
    assert call(acc=None) == binding.ERR_INVALID_ARG
    assert call(r=ctypes.c_void_p((1 << 20) + 4)) == binding.ERR_INVALID_ARG  # r_cut: 8-byte aligned
    assert call(s=ctypes.c_void_p((1 << 20) + 2)) == binding.ERR_INVALID_ARG
    assert call(st=ctypes.c_void_p((1 << 20) + 1)) == binding.ERR_INVALID_ARG
    assert call(G=0, N=0) == binding.OK


def test_verify_scd_host_checks(binding):
    """spec_verify_scd's argument errors return before any launch (fake,
    never dereferenced pointers)."""
    f = binding._lib.spec_verify_scd
    fake = ctypes.c_void_p(1 << 20)
    ws = binding.workspace_size(4, 3, 1024, binding.DTYPE_F32, binding.MODE_SAMPLE)
    def call(B=4, K=3, V=1024, dtype=binding.DTYPE_F32, T=1.0, alpha=0.1, t=fake, a=fake, x=fake,
             u=fake, nbytes=ws):
        return f(t, a, x, u, B, K, V, dtype, T, alpha, fake, fake, fake, nbytes, None,
                 None, None, None, None)
    assert call(B=-1) == binding.ERR_INVALID_ARG
    assert call(V=0) == binding.ERR_INVALID_ARG
    assert call(dtype=5) == binding.ERR_INVALID_ARG
    assert call(T=0.0) == binding.ERR_INVALID_ARG
    for bad in (-0.5, 1.5, float("nan")):
        assert call(alpha=bad) == binding.ERR_INVALID_ARG
    assert call(a=None) == binding.ERR_INVALID_ARG
    assert call(t=None) == binding.ERR_INVALID_ARG
    assert call(x=None) == binding.ERR_INVALID_ARG
    assert call(u=None) == binding.ERR_INVALID_ARG
    assert call(nbytes=64) == binding.ERR_INVALID_ARG
    assert call(K=binding.MAX_K + 1) == binding.ERR_UNSUPPORTED
    wsu = binding.workspace_size(4, 3, 1001, binding.DTYPE_F32, binding.MODE_SAMPLE)
    assert call(V=1001, nbytes=wsu) == binding.ERR_UNSUPPORTED  # rows not 16-byte multiples
    wsl = binding.workspace_size(4, 3, 1 << 22, binding.DTYPE_F32, binding.MODE_SAMPLE)
    assert call(V=1 << 22, nbytes=wsl) == binding.ERR_UNSUPPORTED  # a row pair beyond 8 CTAs
    assert call(B=0) == binding.OK


def test_c_program_uses_the_boundary_without_python(binding, tmp_path):
    """A plain C11 program includes the header and links the library (no
    torch, no Python): it builds with -Wall -Werror and its host-side checks
    pass without a GPU."""
    src = os.path.join(os.path.dirname(__file__), "c_abi", "abi_check.c")
    exe = str(tmp_path / "abi_check")
    libdir = os.path.dirname(binding.LIB_PATH)
    cc = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I",
                         os.path.dirname(HEADER), src, "-L", libdir, "-lspecverify",
                         "-Wl,-rpath," + libdir, "-o", exe], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, (run.returncode, run.stderr)
    assert "all checks passed" in run.stdout


def test_debug_variant_builds_with_the_same_exports(binding):
    """The -DSPEC_DEBUG test variant (index checks that report instead of
    faulting) builds from the same sources and exports the same entry points;
    the optional NVTX ranges (-DSPEC_NVTX) compile."""
    import subprocess
    from draft_verify_acceptance_gb300 import build
    lib = build.build(debug=True)
    assert lib.endswith("libspecverify_debug.so")
    dbg = ctypes.CDLL(lib)
    for n in binding.EXPORTS:
        assert hasattr(dbg, n), n
    src = os.path.join(build.CSRC, "spec_verify.cu")
    r = subprocess.run([build._nvcc(), "-std=c++17", *build.ARCH, "-DSPEC_NVTX", "-c", src,
                        "-o", os.devnull, "-I", os.path.join(build.ROOT, "include")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
