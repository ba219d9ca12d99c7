"""ctypes binding of libspecverify.so -- argument marshalling only.

Every step of the verify path runs in the library's CUDA kernels; this module
checks tensor dtypes, shapes, devices and contiguity, owns a zero-filled
workspace per (device, stream), and passes raw pointers plus the current
CUDA stream through the C ABI.  There is no CPU fallback: if the library is
missing or a tensor is not on a CUDA device, it raises.
"""
import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

MODE_SAMPLE = 0
MODE_GREEDY = 1
MODE_SAMPLE_EARLY_EXIT = 2
DTYPE_F32 = 0
DTYPE_BF16 = 1
MAX_K = 64
MAX_V = 1 << 22

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_CUDA = 3
ERR_SCRATCH_LIMIT = 4
STATIC_SCRATCH_BYTES = 1 << 20

DATA_TOKEN_RANGE = 1
DATA_NONFINITE_LOGIT = 2
DATA_UNIFORM_RANGE = 4
DEVICE_WAIT_TIMEOUT = 8
DATA_NONFINITE_SCORE = 16
FLAG_RATIO = 1
FLAG_CDF = 2

EXPORTS = ("spec_verify", "spec_verify_ex", "spec_verify_workspace_size", "spec_status_string",
           "spec_verify_static", "spec_draft_sample", "spec_rejection_cut", "spec_verify_scd",
           "spec_set_wait_limit")


class SpecVerifyError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {status_string(code)} (code {code})")
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with draft_verify_acceptance_gb300.build.build() "
            "(nvcc for sm_103a); there is no fallback implementation")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.spec_verify_workspace_size.restype = Z
    lib.spec_verify_workspace_size.argtypes = [I, I, I, I, I]
    lib.spec_verify.restype = I
    lib.spec_verify.argtypes = [P, P, P, P, I, I, I, I, F, I, P, P, P, Z, P]
    lib.spec_verify_ex.restype = I
    lib.spec_verify_ex.argtypes = [P, P, P, P, I, I, I, I, F, I, P, P, P, Z, P, P, P, P, P]
    lib.spec_verify_static.restype = I
    lib.spec_verify_static.argtypes = [P, P, P, P, I, I, I, I, F, I, P, P, P]
    lib.spec_draft_sample.restype = I
    lib.spec_draft_sample.argtypes = [P, P, I, I, I, F, P, P, P, Z, P, P]
    lib.spec_verify_scd.restype = I
    lib.spec_verify_scd.argtypes = [P, P, P, P, I, I, I, I, F, ctypes.c_double, P, P, P, Z, P,
                                    P, P, P, P]
    lib.spec_rejection_cut.restype = I
    lib.spec_rejection_cut.argtypes = [P, I, I, ctypes.c_double, P, P, P, P, P]
    lib.spec_set_wait_limit.restype = I
    lib.spec_set_wait_limit.argtypes = [ctypes.c_uint]
    lib.spec_status_string.restype = ctypes.c_char_p
    lib.spec_status_string.argtypes = [I]
    return lib


_lib = _load()
_ws_lock = threading.Lock()
_ws_cache = {}


def status_string(code: int) -> str:
    return _lib.spec_status_string(int(code)).decode()


def set_wait_limit(microseconds: int) -> None:
    """Bound (microseconds; 0 = the default 2 s) on a kernel's waits for work
    of other thread blocks; past it the kernel stops and reports
    DEVICE_WAIT_TIMEOUT in the status word (spec_set_wait_limit)."""
    _lib.spec_set_wait_limit(int(microseconds))


def workspace_size(B: int, K: int, V: int, dtype: int, mode: int) -> int:
    return int(_lib.spec_verify_workspace_size(B, K, V, dtype, mode))


def workspace_for(device: torch.device, stream: torch.cuda.Stream, nbytes: int) -> torch.Tensor:
    """A zero-filled workspace of at least ``nbytes`` for this device and
    stream.  The kernels leave it zero-filled after every call, so it is
    reused; each stream gets its own so concurrent calls never share one."""
    key = (device.index, stream.cuda_stream)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < nbytes:
            with torch.cuda.stream(stream):
                ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
        return ws


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtypes, shape, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _mode(mode):
    if isinstance(mode, str):
        return {"sample": MODE_SAMPLE, "greedy": MODE_GREEDY,
                "sample_early_exit": MODE_SAMPLE_EARLY_EXIT}[mode]
    return int(mode)


def _call(target, draft, tokens, uniforms, temperature, mode, debug, stream, workspace,
          out=None):
    mode = _mode(mode)
    if target is None or target.dim() != 3:
        raise ValueError("target must be [B, K+1, V]")
    device = target.device
    B, K1, V = target.shape
    K = K1 - 1
    _check(target, "target", (torch.float32, torch.bfloat16), (B, K1, V), device)
    dt = DTYPE_BF16 if target.dtype == torch.bfloat16 else DTYPE_F32
    sample = mode != MODE_GREEDY
    if K > 0:
        _check(tokens, "tokens", (torch.int32,), (B, K), device)
    if sample:
        if K > 0:
            _check(draft, "draft", (target.dtype,), (B, K, V), device)
        _check(uniforms, "uniforms", (torch.float32,), (B, K1), device)
    stream = stream or torch.cuda.current_stream(device)
    if out is not None:
        acc, out = out
        _check(acc, "accepted_len", (torch.int32,), (B,), device)
        _check(out, "out_tokens", (torch.int32,), (B, K1), device)
    else:
        acc = torch.empty(B, dtype=torch.int32, device=device)
        out = torch.empty((B, K1), dtype=torch.int32, device=device)
    need = workspace_size(B, K, V, dt, mode)
    if need == 0 and B > 0:
        raise SpecVerifyError(ERR_UNSUPPORTED if K > MAX_K or V > MAX_V else ERR_INVALID_ARG,
                              "workspace size")
    ws = workspace if workspace is not None else workspace_for(device, stream, need)
    extras = None
    with torch.cuda.device(device):
        if debug:
            p_at = torch.zeros((B, K), dtype=torch.float32, device=device)
            q_at = torch.zeros((B, K), dtype=torch.float32, device=device)
            flags = torch.zeros(B, dtype=torch.int32, device=device)
            status = torch.zeros(1, dtype=torch.int32, device=device)
            rc = _lib.spec_verify_ex(
                _ptr(target), _ptr(draft if sample else None), _ptr(tokens if K > 0 else None),
                _ptr(uniforms if sample else None), B, K, V, dt, float(temperature), mode,
                _ptr(acc), _ptr(out), _ptr(ws), ws.numel(), ctypes.c_void_p(stream.cuda_stream),
                _ptr(p_at), _ptr(q_at), _ptr(flags), _ptr(status))
            extras = dict(p_at=p_at, q_at=q_at, flags=flags, status=status)
        else:
            rc = _lib.spec_verify(
                _ptr(target), _ptr(draft if sample else None), _ptr(tokens if K > 0 else None),
                _ptr(uniforms if sample else None), B, K, V, dt, float(temperature), mode,
                _ptr(acc), _ptr(out), _ptr(ws), ws.numel(), ctypes.c_void_p(stream.cuda_stream))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_verify")
    return acc, out, extras


def verify(target, draft=None, tokens=None, uniforms=None, temperature=1.0, mode="sample",
           *, stream=None, workspace=None, out=None):
    """One verify step on the GPU.

    target [B, K+1, V] and draft [B, K, V] (float32 or bfloat16), tokens [B, K]
    int32, uniforms [B, K+1] float32, all CUDA tensors on one device.  Returns
    (accepted_len [B], out_tokens [B, K+1]) as int32 CUDA tensors, queued on
    ``stream`` (default: the current stream).  ``out`` may give preallocated
    (accepted_len, out_tokens) tensors to write into; ``workspace`` a
    zero-filled uint8 CUDA tensor of at least ``workspace_size(...)`` bytes.

    Host (CPU) tensors are accepted too: they are copied to the current CUDA
    device (asynchronously when pinned), verified there, and the results are
    copied back to the host before returning.
    """
    if target is not None and not target.is_cuda:
        return _verify_host(target, draft, tokens, uniforms, temperature, mode, stream)
    acc, res, _ = _call(target, draft, tokens, uniforms, temperature, mode, False, stream,
                        workspace, out)
    return acc, res


def verify_ex(target, draft=None, tokens=None, uniforms=None, temperature=1.0, mode="sample",
              *, stream=None, workspace=None):
    """``verify`` plus diagnostics: a dict with accepted_len, out_tokens,
    p_at / q_at [B, K] (p_i(x_i), q_i(x_i)), flags [B] (boundary flags) and
    status [1] (OR of data-error bits)."""
    acc, out, ex = _call(target, draft, tokens, uniforms, temperature, mode, True, stream, workspace)
    ex.update(accepted_len=acc, out_tokens=out)
    return ex


def draft_sample(logits, uniforms, temperature=1.0, *, stream=None, workspace=None, out=None,
                 debug=False):
    """The drafter's sampling step on the GPU: for each row of ``logits``
    ([..., V], float32 or bfloat16, CUDA, 16-byte aligned rows) draw x from
    softmax(row / T) by inverse CDF with the matching uniform ([...] float32).
    Returns (tokens int32 [...], q_at float32 [...] = q(x)), plus the status
    word when ``debug``, queued on ``stream``; ``out`` may give preallocated
    (tokens, q_at)."""
    if logits is None or logits.dim() < 1:
        raise ValueError("logits must be [..., V]")
    device = logits.device
    V = logits.shape[-1]
    R = logits.numel() // V if V else 0
    _check(logits, "logits", (torch.float32, torch.bfloat16), tuple(logits.shape), device)
    _check(uniforms, "uniforms", (torch.float32,), tuple(logits.shape[:-1]), device)
    dt = DTYPE_BF16 if logits.dtype == torch.bfloat16 else DTYPE_F32
    stream = stream or torch.cuda.current_stream(device)
    if out is not None:
        tokens, q_at = out
        _check(tokens, "tokens", (torch.int32,), tuple(logits.shape[:-1]), device)
        _check(q_at, "q_at", (torch.float32,), tuple(logits.shape[:-1]), device)
    else:
        tokens = torch.empty(logits.shape[:-1], dtype=torch.int32, device=device)
        q_at = torch.empty(logits.shape[:-1], dtype=torch.float32, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device) if debug else None
    need = workspace_size(R, 0, V, dt, MODE_SAMPLE)
    if need == 0 and R > 0:
        raise SpecVerifyError(ERR_UNSUPPORTED if V > MAX_V else ERR_INVALID_ARG, "workspace size")
    ws = workspace if workspace is not None else workspace_for(device, stream, need)
    with torch.cuda.device(device):
        rc = _lib.spec_draft_sample(_ptr(logits), _ptr(uniforms), R, V, dt, float(temperature),
                                    _ptr(tokens), _ptr(q_at), _ptr(ws), ws.numel(),
                                    ctypes.c_void_p(stream.cuda_stream), _ptr(status))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_draft_sample")
    return (tokens, q_at, status) if debug else (tokens, q_at)


def verify_scd(target, amateur, tokens, uniforms, temperature=1.0, alpha=0.1, *, stream=None,
               workspace=None, out=None, debug=False):
    """Speculative contrastive decoding's verify step on the GPU: target and
    amateur [B, K+1, V] (float32 or bfloat16, CUDA, 16-byte aligned rows),
    tokens [B, K] int32 (drawn from the amateur), uniforms [B, K+1] float32,
    alpha the plausibility cut of the contrastive head.  Returns
    (accepted_len, out_tokens), or with ``debug`` a dict that adds p_at
    (P_n(x_i)), q_at, flags and status; queued on ``stream``."""
    if target is None or target.dim() != 3:
        raise ValueError("target must be [B, K+1, V]")
    device = target.device
    B, K1, V = target.shape
    K = K1 - 1
    _check(target, "target", (torch.float32, torch.bfloat16), (B, K1, V), device)
    _check(amateur, "amateur", (target.dtype,), (B, K1, V), device)
    if K > 0:
        _check(tokens, "tokens", (torch.int32,), (B, K), device)
    _check(uniforms, "uniforms", (torch.float32,), (B, K1), device)
    dt = DTYPE_BF16 if target.dtype == torch.bfloat16 else DTYPE_F32
    stream = stream or torch.cuda.current_stream(device)
    if out is not None:
        acc, res = out
        _check(acc, "accepted_len", (torch.int32,), (B,), device)
        _check(res, "out_tokens", (torch.int32,), (B, K1), device)
    else:
        acc = torch.empty(B, dtype=torch.int32, device=device)
        res = torch.empty((B, K1), dtype=torch.int32, device=device)
    need = workspace_size(B, K, V, dt, MODE_SAMPLE)
    if need == 0 and B > 0:
        raise SpecVerifyError(ERR_UNSUPPORTED if K > MAX_K or V > MAX_V else ERR_INVALID_ARG,
                              "workspace size")
    ws = workspace if workspace is not None else workspace_for(device, stream, need)
    ex = None
    if debug:
        ex = dict(p_at=torch.zeros((B, K), dtype=torch.float32, device=device),
                  q_at=torch.zeros((B, K), dtype=torch.float32, device=device),
                  flags=torch.zeros(B, dtype=torch.int32, device=device),
                  status=torch.zeros(1, dtype=torch.int32, device=device))
    with torch.cuda.device(device):
        rc = _lib.spec_verify_scd(
            _ptr(target), _ptr(amateur), _ptr(tokens if K > 0 else None), _ptr(uniforms), B, K, V,
            dt, float(temperature), float(alpha), _ptr(acc), _ptr(res), _ptr(ws), ws.numel(),
            ctypes.c_void_p(stream.cuda_stream), _ptr(ex and ex["p_at"]), _ptr(ex and ex["q_at"]),
            _ptr(ex and ex["flags"]), _ptr(ex and ex["status"]))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_verify_scd")
    if debug:
        ex.update(accepted_len=acc, out_tokens=res)
        return ex
    return acc, res


def rejection_cut(scores, alpha, *, stream=None, out=None, debug=False):
    """Speculative Rejection's cut on the GPU: for each prompt (row of
    ``scores``, [G, N] float32, CUDA) r_cut = the alpha-quantile of its N
    reward scores, and the indices scoring at least r_cut.  Returns (r_cut
    float64 [G], n_accepted int32 [G], accepted int32 [G, N]: kept indices in
    ascending order then -1), plus the status word when ``debug``, queued on
    ``stream``; ``out`` may give those three tensors preallocated."""
    if scores is None or scores.dim() != 2:
        raise ValueError("scores must be [G, N]")
    device = scores.device
    G, N = scores.shape
    _check(scores, "scores", (torch.float32,), (G, N), device)
    stream = stream or torch.cuda.current_stream(device)
    if out is not None:
        r_cut, n_acc, acc = out
        _check(r_cut, "r_cut", (torch.float64,), (G,), device)
        _check(n_acc, "n_accepted", (torch.int32,), (G,), device)
        _check(acc, "accepted", (torch.int32,), (G, N), device)
    else:
        r_cut = torch.empty(G, dtype=torch.float64, device=device)
        n_acc = torch.empty(G, dtype=torch.int32, device=device)
        acc = torch.empty((G, N), dtype=torch.int32, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device) if debug else None
    with torch.cuda.device(device):
        rc = _lib.spec_rejection_cut(_ptr(scores), G, N, float(alpha), _ptr(r_cut), _ptr(n_acc),
                                     _ptr(acc), ctypes.c_void_p(stream.cuda_stream), _ptr(status))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_rejection_cut")
    return (r_cut, n_acc, acc, status) if debug else (r_cut, n_acc, acc)


def _verify_host(target, draft, tokens, uniforms, temperature, mode, stream):
    device = torch.device("cuda", torch.cuda.current_device())
    stream = stream or torch.cuda.current_stream(device)
    with torch.cuda.stream(stream):
        dev = [None if t is None else t.to(device, non_blocking=True)
               for t in (target, draft, tokens, uniforms)]
        acc, out, _ = _call(*dev, temperature, mode, False, stream, None)
        acc_h = torch.empty(acc.shape, dtype=acc.dtype, pin_memory=True)
        out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        acc_h.copy_(acc, non_blocking=True)
        out_h.copy_(out, non_blocking=True)
    stream.synchronize()
    return acc_h, out_h
