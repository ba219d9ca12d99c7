"""CPU oracle of the draft-then-verify acceptance step (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg import this package.  The CUDA
library never imports, links or calls it, and it never calls the CUDA library.

The arithmetic lives in ``spec_oracle.c`` (plain C, IEEE double); this module
only marshals numpy arrays to pointers.
"""
import ctypes
import os

import numpy as np

from . import build as _build

MODE_SAMPLE = 0
MODE_GREEDY = 1
DTYPE_F32 = 0
DTYPE_BF16 = 1
VARIANT_EXACT = 0
VARIANT_LITERAL_TARGET = 1  # negative control: correction drawn from p_n

DATA_TOKEN = 1
DATA_LOGIT = 2
DATA_UNIFORM = 4
DATA_SCORE = 8

FLAG_RATIO = 1
FLAG_CDF = 2
FLAG_TINY_RESIDUAL = 4

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        lib.spec_oracle_verify.restype = ctypes.c_int
        lib.spec_oracle_verify.argtypes = [
            P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P]
        lib.spec_oracle_draft_sample.restype = ctypes.c_int
        lib.spec_oracle_draft_sample.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_double, P, P, P, P]
        lib.spec_oracle_scd_verify.restype = ctypes.c_int
        lib.spec_oracle_scd_verify.argtypes = [
            P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, ctypes.c_double, P, P, P, P, P, P]
        lib.spec_oracle_rejection_cut.restype = ctypes.c_int
        lib.spec_oracle_rejection_cut.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                  P, P, P, P]
        lib.spec_oracle_softmax.restype = ctypes.c_int
        lib.spec_oracle_softmax.argtypes = [P, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, P]
        lib.spec_oracle_max_threads.restype = ctypes.c_int
        lib.spec_oracle_set_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a, name):
    """Accept fp32 arrays, or bf16 given as their raw uint16 bit patterns."""
    if a is None:
        return None, None
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, DTYPE_F32
    if a.dtype == np.uint16:
        return a, DTYPE_BF16
    raise TypeError(f"{name}: expected float32 or uint16 (bf16 bits), got {a.dtype}")


def verify_ref(target, draft, tokens, uniforms, temperature=1.0,
               mode=MODE_SAMPLE, variant=VARIANT_EXACT, want_debug=False):
    """Run the oracle over a batch.

    target [B, K+1, V], draft [B, K, V] (float32 or bf16 bits as uint16),
    tokens [B, K] int32, uniforms [B, K+1] float32.
    Returns a dict: accepted_len [B], out_tokens [B, K+1], status, and with
    ``want_debug`` also p_at / q_at [B, K] (float64) and flags [B] (uint32).
    """
    lib = _load()
    t, dt = _logits(target, "target")
    B, K1, V = t.shape
    K = K1 - 1
    d, ddt = _logits(draft, "draft")
    if d is not None and ddt != dt:
        raise TypeError("target and draft dtypes differ")
    x = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
    u = None if uniforms is None else np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, K + 1)
    n = np.empty(B, np.int32)
    out = np.empty((B, K + 1), np.int32)
    p_at = np.zeros((B, K), np.float64) if want_debug else None
    q_at = np.zeros((B, K), np.float64) if want_debug else None
    flags = np.zeros(B, np.uint32) if want_debug else None
    status = ctypes.c_int32(0)
    rc = lib.spec_oracle_verify(_ptr(t), _ptr(d), _ptr(x), _ptr(u), B, K, V, dt,
                                float(temperature), mode, variant, _ptr(n), _ptr(out),
                                _ptr(p_at), _ptr(q_at), _ptr(flags),
                                ctypes.byref(status))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    res = {"accepted_len": n, "out_tokens": out, "status": status.value}
    if want_debug:
        res.update(p_at=p_at, q_at=q_at, flags=flags)
    return res


def scd_verify_ref(target, amateur, tokens, uniforms, temperature=1.0, alpha=0.1,
                   want_debug=False):
    """Speculative contrastive decoding over a batch: target and amateur
    [B, K+1, V] (float32, or bf16 bits as uint16), tokens [B, K] int32,
    uniforms [B, K+1] float32, alpha the plausibility cut.  Returns the same
    dict as verify_ref (p_at is P_n(x_i), q_at the amateur's q(x_i))."""
    lib = _load()
    t, dt = _logits(target, "target")
    B, K1, V = t.shape
    K = K1 - 1
    a, adt = _logits(amateur, "amateur")
    if adt != dt or a.shape != t.shape:
        raise TypeError("target and amateur must match in dtype and shape")
    x = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
    u = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, K + 1)
    n = np.empty(B, np.int32)
    out = np.empty((B, K + 1), np.int32)
    p_at = np.zeros((B, K), np.float64) if want_debug else None
    q_at = np.zeros((B, K), np.float64) if want_debug else None
    flags = np.zeros(B, np.uint32) if want_debug else None
    status = ctypes.c_int32(0)
    rc = lib.spec_oracle_scd_verify(_ptr(t), _ptr(a), _ptr(x), _ptr(u), B, K, V, dt,
                                    float(temperature), float(alpha), _ptr(n), _ptr(out),
                                    _ptr(p_at), _ptr(q_at), _ptr(flags), ctypes.byref(status))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    res = {"accepted_len": n, "out_tokens": out, "status": status.value}
    if want_debug:
        res.update(p_at=p_at, q_at=q_at, flags=flags)
    return res


def draft_sample_ref(logits, uniforms, temperature=1.0):
    """The drafter's sampling step: x ~ softmax(row / T) by inverse CDF with
    one uniform per row.  logits [..., V] (float32 or bf16 bits as uint16),
    uniforms [...] float32.  Returns tokens (int32), q_at = q(x) (float64),
    flags (uint32) shaped like the uniforms, and status."""
    lib = _load()
    t, dt = _logits(logits, "logits")
    V = t.shape[-1]
    R = t.size // V
    u = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(-1)
    if u.size != R:
        raise ValueError("one uniform per row")
    tok = np.empty(R, np.int32)
    q = np.empty(R, np.float64)
    flags = np.empty(R, np.uint32)
    status = ctypes.c_int32(0)
    rc = lib.spec_oracle_draft_sample(_ptr(t), _ptr(u), R, V, dt, float(temperature), _ptr(tok),
                                      _ptr(q), _ptr(flags), ctypes.byref(status))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    shape = t.shape[:-1]
    return {"tokens": tok.reshape(shape), "q_at": q.reshape(shape),
            "flags": flags.reshape(shape), "status": status.value}


def rejection_cut_ref(scores, alpha):
    """Speculative Rejection's cut over G prompts of N reward scores each.
    scores [G, N] float32, alpha in [0, 1].  Returns r_cut [G] (float64),
    n_accepted [G] (int32), accepted [G, N] (int32, ascending indices of the
    kept sequences, then -1) and status."""
    lib = _load()
    s = np.ascontiguousarray(scores, dtype=np.float32)
    if s.ndim != 2:
        raise ValueError("scores must be [G, N]")
    G, N = s.shape
    r = np.empty(G, np.float64)
    n = np.empty(G, np.int32)
    acc = np.empty((G, N), np.int32)
    status = ctypes.c_int32(0)
    rc = lib.spec_oracle_rejection_cut(_ptr(s), G, N, float(alpha), _ptr(r), _ptr(n), _ptr(acc),
                                       ctypes.byref(status))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return {"r_cut": r, "n_accepted": n, "accepted": acc, "status": status.value}


def softmax_ref(row, temperature=1.0):
    """The oracle's temperature softmax of one row (float64 result)."""
    lib = _load()
    r, dt = _logits(np.asarray(row).reshape(-1), "row")
    p = np.empty(r.shape[0], np.float64)
    rc = lib.spec_oracle_softmax(_ptr(r), r.shape[0], dt, float(temperature), _ptr(p))
    if rc == DATA_LOGIT:
        raise ValueError("row has NaN/+inf or no finite entry")
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return p


def max_threads():
    return _load().spec_oracle_max_threads()


def set_threads(n):
    _load().spec_oracle_set_threads(int(n))
