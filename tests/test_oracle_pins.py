"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests re-derives the oracle's own formulas and compares the
two: each checks a property that holds independently of how the oracle is
written -- the exact output distribution (brute force and chi-square), the
equivalence of greedy verification with plain greedy decoding, the worked
examples printed on the pages, the library softmax, and the accept rule's
special cases.  A negative control shows the exactness checks do catch the
literal "correction sampled from the target" reading.
"""
import itertools
import json
import os
import zlib

import numpy as np
import pytest
import torch
from scipy import stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# softmax: a special case that reduces to a library routine
# --------------------------------------------------------------------------
@pytest.mark.parametrize("V", [1, 2, 7, 1000, 32000])
@pytest.mark.parametrize("T", [1.0, 0.7, 2.3])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_softmax_matches_library(V, T, dtype):
    g = torch.Generator().manual_seed(V * 7 + int(T * 10))
    x = torch.randn(V, generator=g) * 4.0
    if V > 3:
        x[1] = float("-inf")
    if dtype == "bf16":
        xb = x.to(torch.bfloat16)
        arr = xb.view(torch.int16).numpy().view(np.uint16)
        xd = xb.double()
    else:
        arr = x.numpy()
        xd = x.double()
    p = oracle.softmax_ref(arr, T)
    ref = torch.softmax(xd / T, dim=0).numpy()
    np.testing.assert_allclose(p, ref, rtol=1e-12, atol=1e-15)
    assert abs(p.sum() - 1.0) < 1e-12


def test_softmax_rejects_nan_and_inf():
    with pytest.raises(ValueError):
        oracle.softmax_ref(np.array([0.0, np.nan, 1.0], np.float32))
    with pytest.raises(ValueError):
        oracle.softmax_ref(np.array([0.0, np.inf, 1.0], np.float32))
    with pytest.raises(ValueError):
        oracle.softmax_ref(np.array([-np.inf, -np.inf], np.float32))


# --------------------------------------------------------------------------
# exactness by brute force (V <= 4, K <= 2)
# --------------------------------------------------------------------------
def _tables(V, K, seed, T):
    """Prefix-indexed logit tables: target rows for prefixes of length 0..K,
    draft rows for prefixes of length 0..K-1.  Some tokens get -inf."""
    rng = np.random.default_rng(seed)
    tgt, drf = {}, {}
    for L in range(K + 1):
        for pre in itertools.product(range(V), repeat=L):
            t = rng.normal(0, 1.5, V)
            if V > 2 and rng.random() < 0.3:
                t[rng.integers(V)] = -np.inf
            tgt[pre] = t.astype(np.float32)
            if L < K:
                d = t + rng.normal(0, 1.0, V)
                d[~np.isfinite(d)] = rng.normal(0, 1.0)
                if V > 2 and rng.random() < 0.3:
                    d[rng.integers(V)] = -np.inf
                if not np.isfinite(d).any():
                    d[0] = 0.0
                drf[pre] = d.astype(np.float32)
    return tgt, drf


def _probs(logits, T):
    return torch.softmax(torch.from_numpy(logits.astype(np.float64)) / T, 0).numpy()


def _cells(cuts):
    pts = sorted(set([0.0, 1.0] + [c for c in cuts if 0.0 < c < 1.0]))
    return [(a, b) for a, b in zip(pts[:-1], pts[1:]) if b > a]


def _exact_joint(V, K, seed, T, variant):
    """Joint law of the K+1 tokens obtained by one verify step followed by
    plain target sampling of the remaining positions, integrated exactly over
    the uniforms.  The uniforms' cells come from the breakpoints where any
    correct sampler may change its answer; the oracle is probed at several
    points per cell and must answer the same at all of them."""
    tgt, drf = _tables(V, K, seed, T)
    P = {k: _probs(v, T) for k, v in tgt.items()}
    Q = {k: _probs(v, T) for k, v in drf.items()}
    rows_t, rows_d, toks, us, meta = [], [], [], [], []
    fracs = (0.13, 0.5, 0.87)
    for x in itertools.product(range(V), repeat=K):
        w = 1.0
        for i in range(K):
            w *= Q[x[:i]][x[i]]
        if w == 0.0:
            continue
        # breakpoints of the accept tests
        acc_cells = []
        for i in range(K):
            p, q = P[x[:i]][x[i]], Q[x[:i]][x[i]]
            acc_cells.append(_cells([min(1.0, p / q)]))
        # breakpoints of the final draw: CDF points of every row it may use
        # (a superset of cuts is harmless: it only refines the cells)
        cuts = []
        for n in range(K + 1):
            cuts.extend(np.cumsum(P[x[:n]]))
            if n < K:
                res = np.maximum(0.0, P[x[:n]] - Q[x[:n]])
                if res.sum() > 0:
                    cuts.extend(np.cumsum(res) / res.sum())
        last_cells = _cells(cuts)
        t_rows = np.stack([tgt[x[:i]] for i in range(K + 1)])
        d_rows = np.stack([drf[x[:i]] for i in range(K)]) if K else np.zeros((0, V), np.float32)
        for combo in itertools.product(*(acc_cells + [last_cells])):
            m = w
            for a, b in combo:
                m *= b - a
            if m == 0.0:
                continue
            for f in fracs:
                u = np.array([a + f * (b - a) for a, b in combo], np.float32)
                # keep the probe strictly inside its cell after fp32 rounding
                u = np.array([min(max(v, np.nextafter(np.float32(a), np.float32(2))),
                                  np.nextafter(np.float32(b), np.float32(-1)))
                              for v, (a, b) in zip(u, combo)], np.float32)
                rows_t.append(t_rows)
                rows_d.append(d_rows)
                toks.append(np.array(x, np.int32))
                us.append(u)
                meta.append((x, combo, m, f))
    res = oracle.verify_ref(np.stack(rows_t), np.stack(rows_d), np.stack(toks).reshape(len(toks), K),
                            np.stack(us), T, oracle.MODE_SAMPLE, variant)
    assert res["status"] == 0
    joint = np.zeros((V,) * (K + 1))
    seen = {}
    for j, (x, combo, m, f) in enumerate(meta):
        n = int(res["accepted_len"][j])
        emitted = tuple(int(v) for v in res["out_tokens"][j][: n + 1])
        key = (x, combo)
        if key in seen:
            assert seen[key] == emitted, "oracle answer changes inside one cell"
            continue
        seen[key] = emitted
        # finish the sequence with plain target sampling
        for rest in itertools.product(range(V), repeat=K - n):
            y = emitted + rest
            pr = m
            for k in range(n + 1, K + 1):
                pr *= P[y[:k]][y[k]]
            joint[y] += pr
    target_joint = np.zeros_like(joint)
    for y in itertools.product(range(V), repeat=K + 1):
        pr = 1.0
        for k in range(K + 1):
            pr *= P[y[:k]][y[k]]
        target_joint[y] = pr
    return joint, target_joint


@pytest.mark.parametrize("V,K,seed,T", [(2, 1, 1, 1.0), (3, 1, 2, 0.8), (3, 2, 3, 1.0),
                                        (4, 2, 4, 1.3), (4, 1, 5, 0.7), (4, 2, 6, 1.0),
                                        (3, 0, 7, 1.0)])
def test_brute_force_output_law_is_the_target_law(V, K, seed, T):
    joint, target = _exact_joint(V, K, seed, T, oracle.VARIANT_EXACT)
    assert abs(joint.sum() - 1.0) < 1e-12
    np.testing.assert_allclose(joint, target, rtol=0, atol=1e-12)


@pytest.mark.parametrize("V,K,seed", [(3, 1, 2), (4, 2, 4)])
def test_brute_force_catches_literal_target_correction(V, K, seed):
    """Negative control: drawing the correction from p_n (the literal wording
    of the rejection-sampling page's step 4) is not exact."""
    joint, target = _exact_joint(V, K, seed, 1.0, oracle.VARIANT_LITERAL_TARGET)
    assert np.abs(joint - target).max() > 1e-3


# --------------------------------------------------------------------------
# exactness by sampling: chi-square over 10^6 seeded trials, V = 8
# --------------------------------------------------------------------------
def _mc_batch(K, n_trials, seed, T=1.0):
    V = 8
    rng = np.random.default_rng(seed)
    tgt, drf = {}, {}
    for L in range(K + 1):
        for pre in itertools.product(range(V), repeat=L):
            t = rng.normal(0, 1.5, V).astype(np.float32)
            tgt[pre] = t
            if L < K:
                drf[pre] = (t + rng.normal(0, 1.5, V)).astype(np.float32)
    Q = {k: _probs(v, T) for k, v in drf.items()}
    x = np.zeros((n_trials, K), np.int32)
    for i in range(K):
        for pre in itertools.product(range(V), repeat=i):
            sel = np.all(x[:, :i] == np.array(pre, np.int32), axis=1) if i else np.ones(n_trials, bool)
            cnt = int(sel.sum())
            if cnt:
                x[sel, i] = rng.choice(V, size=cnt, p=Q[pre])
    t_rows = np.empty((n_trials, K + 1, V), np.float32)
    d_rows = np.empty((n_trials, K, V), np.float32)
    for i in range(K + 1):
        for pre in itertools.product(range(V), repeat=i):
            sel = np.all(x[:, :i] == np.array(pre, np.int32), axis=1) if i else np.ones(n_trials, bool)
            t_rows[sel, i] = tgt[pre]
            if i < K:
                d_rows[sel, i] = drf[pre]
    u = rng.random((n_trials, K + 1), dtype=np.float32)
    return tgt, drf, t_rows, d_rows, x, u


@pytest.mark.parametrize("K", [1, 2])
def test_chi_square_first_token_follows_target(K):
    n = 1_000_000
    tgt, drf, t, d, x, u = _mc_batch(K, n, seed=11 + K)
    res = oracle.verify_ref(t, d, x, u, 1.0)
    first = res["out_tokens"][:, 0]
    counts = np.bincount(first, minlength=8)
    p0 = _probs(tgt[()], 1.0)
    chi2, pval = stats.chisquare(counts, n * p0)
    assert pval > 1e-3, (chi2, pval)
    # negative control: the literal reading is rejected decisively
    bad = oracle.verify_ref(t, d, x, u, 1.0, variant=oracle.VARIANT_LITERAL_TARGET)
    counts_bad = np.bincount(bad["out_tokens"][:, 0], minlength=8)
    _, pval_bad = stats.chisquare(counts_bad, n * p0)
    assert pval_bad < 1e-12
    # acceptance rate at position 0 is sum_x min(p, q)
    q0 = _probs(drf[()], 1.0)
    beta = np.minimum(p0, q0).sum()
    acc = (res["accepted_len"] >= 1).mean()
    assert abs(acc - beta) < 5 * np.sqrt(beta * (1 - beta) / n)


def test_chi_square_second_token_given_first():
    """K = 2: among trials whose first emitted token is a, the second emitted
    token (when there is one, or the next target draw) follows p(. | a).
    Trials that stopped at n = 0 are completed with a fresh target draw."""
    n = 1_000_000
    K = 2
    tgt, drf, t, d, x, u = _mc_batch(K, n, seed=29)
    res = oracle.verify_ref(t, d, x, u, 1.0)
    out, nacc = res["out_tokens"], res["accepted_len"]
    rng = np.random.default_rng(99)
    second = out[:, 1].copy()
    stop0 = nacc == 0
    for a in range(8):
        sel = stop0 & (out[:, 0] == a)
        if sel.any():
            second[sel] = rng.choice(8, size=int(sel.sum()), p=_probs(tgt[(a,)], 1.0))
    for a in range(8):
        sel = out[:, 0] == a
        if sel.sum() < 2000:
            continue
        counts = np.bincount(second[sel], minlength=8)
        pa = _probs(tgt[(a,)], 1.0)
        _, pval = stats.chisquare(counts, sel.sum() * pa)
        assert pval > 1e-4, (a, pval)


# --------------------------------------------------------------------------
# greedy: verification reproduces plain greedy decoding exactly
# --------------------------------------------------------------------------
def _toy_logits(prefix, V, seed, ties):
    h = zlib.crc32(np.asarray(prefix, np.int64).tobytes()) ^ seed
    r = np.random.default_rng(h)
    if ties:
        return r.integers(0, 4, V).astype(np.float32)  # many exact ties
    return r.normal(0, 2, V).astype(np.float32)


@pytest.mark.parametrize("V,K,ties,dtype", [(50, 4, False, "f32"), (17, 3, True, "f32"),
                                            (64, 6, False, "bf16"), (9, 8, True, "bf16")])
def test_greedy_verify_equals_plain_greedy_decoding(V, K, ties, dtype):
    seed = V * 31 + K

    def logits(prefix):
        x = _toy_logits(prefix, V, seed, ties)
        if dtype == "bf16":
            return torch.from_numpy(x).to(torch.bfloat16)
        return torch.from_numpy(x)

    def raw(t):
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    ctx0 = [1, 2, 3]
    m = 80
    plain = list(ctx0)
    while len(plain) < len(ctx0) + m:
        plain.append(int(np.argmax(logits(plain).float().numpy())))
    rng = np.random.default_rng(seed)
    spec = list(ctx0)
    calls = 0
    while len(spec) < len(ctx0) + m:
        # a noisy drafter: right most of the time, wrong sometimes
        drafts, c = [], list(spec)
        for _ in range(K):
            g = int(np.argmax(logits(c).float().numpy()))
            tok = g if rng.random() < 0.75 else int(rng.integers(V))
            drafts.append(tok)
            c.append(tok)
        rows = np.stack([raw(logits(spec + drafts[:i])) for i in range(K + 1)])[None]
        res = oracle.verify_ref(rows, None, np.array([drafts], np.int32), None,
                                mode=oracle.MODE_GREEDY)
        n = int(res["accepted_len"][0])
        emitted = [int(v) for v in res["out_tokens"][0][: n + 1]]
        assert (res["out_tokens"][0][n + 1:] == -1).all()
        assert emitted[:n] == drafts[:n]
        spec.extend(emitted)
        calls += 1
    assert spec[: len(plain)] == plain
    assert calls < m  # more than one token per call on average


def test_greedy_brute_force_all_draft_tuples():
    """Every draft tuple at V = 4, K = 2, with tied maxima in the rows."""
    V, K = 4, 2
    rows = np.array([[1.0, 3.0, 3.0, 0.0], [2.0, 2.0, -np.inf, 1.0], [0.0, 0.0, 0.0, 0.0]],
                    np.float32)
    g = [1, 0, 0]  # lowest index among the maxima
    xs = list(itertools.product(range(V), repeat=K))
    t = np.stack([rows] * len(xs))
    res = oracle.verify_ref(t, None, np.array(xs, np.int32), None, mode=oracle.MODE_GREEDY)
    for j, x in enumerate(xs):
        n = 0
        while n < K and x[n] == g[n]:
            n += 1
        assert res["accepted_len"][j] == n
        assert list(res["out_tokens"][j]) == list(x[:n]) + [g[n]] + [-1] * (K - n)


# --------------------------------------------------------------------------
# the worked examples printed on the pages
# --------------------------------------------------------------------------
def test_worked_example_in_the_bus():
    fx = json.load(open(os.path.join(GOLDEN, "bpd_in_the_bus.json")))
    vocab = fx["vocab"]
    idx = {w: i for i, w in enumerate(vocab)}
    rng = np.random.default_rng(0)
    for case in fx["cases"]:
        K = len(case["draft"])
        rows = rng.normal(0, 0.5, (K + 1, len(vocab))).astype(np.float32)
        for i, w in enumerate(case["target_top1"]):
            rows[i, idx[w]] = 5.0
        res = oracle.verify_ref(rows[None], None, np.array([[idx[w] for w in case["draft"]]], np.int32),
                                None, mode=oracle.MODE_GREEDY)
        assert res["accepted_len"][0] == case["expected_accepted_len"]
        want = [-1 if w is None else idx[w] for w in case["expected_out"]]
        assert list(res["out_tokens"][0]) == want


def test_worked_example_quick_brown_fox():
    fx = json.load(open(os.path.join(GOLDEN, "srs_quick_brown_fox.json")))
    vocab = fx["vocab"]
    idx = {w: i for i, w in enumerate(vocab)}
    with np.errstate(divide="ignore"):
        t = np.log(np.array(fx["target_probs"], np.float64)).astype(np.float32)
        d = np.log(np.array(fx["draft_probs"], np.float64)).astype(np.float32)
    x = np.array([[idx[w] for w in fx["draft"]]], np.int32)
    u = np.array([fx["uniforms"]], np.float32)
    res = oracle.verify_ref(t[None], d[None], x, u, fx["temperature"])
    assert res["accepted_len"][0] == fx["expected_accepted_len"]
    want = [-1 if w is None else idx[w] for w in fx["expected_out"]]
    assert list(res["out_tokens"][0]) == want
    # the outcome does not hinge on the chosen uniforms at positions 2 and K:
    # 'brown' has no target mass and the residual is supported on 'fast' only
    for u2 in (0.0, 0.999):
        for uK in (0.0, 0.5, 0.9999):
            uu = u.copy()
            uu[0, 2], uu[0, 5] = u2, uK
            r2 = oracle.verify_ref(t[None], d[None], x, uu, 1.0)
            assert list(r2["out_tokens"][0]) == want


# --------------------------------------------------------------------------
# the accept rule's special cases and the first-rejection rule
# --------------------------------------------------------------------------
def _one(t, d, x, u, T=1.0):
    return oracle.verify_ref(np.asarray(t, np.float32)[None], np.asarray(d, np.float32)[None],
                             np.asarray(x, np.int32)[None], np.asarray(u, np.float32)[None], T,
                             want_debug=True)


def test_accept_when_target_at_least_draft_for_any_u():
    u_max = np.nextafter(np.float32(1), np.float32(0))
    t = [[2.0, 0.0, 0.0], [0.0, 0.0, 0.0]]   # p(0) > q(0)
    d = [[1.0, 0.0, 0.0]]
    for u0 in (0.0, 0.5, u_max):
        r = _one(t, d, [0], [u0, 0.3])
        assert r["accepted_len"][0] == 1


def test_reject_when_target_has_no_mass_for_any_u():
    t = [[-np.inf, 0.0, 0.0], [0.0, 0.0, 0.0]]
    d = [[3.0, 0.0, 0.0]]
    for u0 in (0.0, 1e-30, 0.5):
        r = _one(t, d, [0], [u0, 0.3])
        assert r["accepted_len"][0] == 0
        assert r["out_tokens"][0][0] in (1, 2)   # never the zero-mass token


def test_accept_when_draft_has_no_mass_but_target_does():
    t = [[0.0, 0.0], [0.0, 0.0]]
    d = [[-np.inf, 0.0]]
    r = _one(t, d, [0], [0.999, 0.3])
    assert r["accepted_len"][0] == 1


def test_accept_probability_threshold_is_p_over_q():
    # V = 2: p = (1/2, 1/2), q = (3/4, 1/4)  =>  p(0)/q(0) = 2/3
    t = [[0.0, 0.0], [0.0, 0.0]]
    d = [[np.log(3.0), 0.0]]
    r = _one(t, d, [0], [0.6666, 0.3])
    assert r["accepted_len"][0] == 1
    r = _one(t, d, [0], [0.6668, 0.3])
    assert r["accepted_len"][0] == 0
    # the residual max(0, p - q) = (0, 1/4): token 1 for every u_K
    for uK in (0.0, 0.5, 0.99):
        r = _one(t, d, [0], [0.9, uK])
        assert list(r["out_tokens"][0]) == [1, -1]


def test_rows_after_first_rejection_do_not_matter():
    rng = np.random.default_rng(5)
    B, K, V = 200, 6, 30
    t = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    d = (t[:, :K] + rng.normal(0, 2, (B, K, V))).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    base = oracle.verify_ref(t, d, x, u)
    n = base["accepted_len"]
    assert ((n >= 0) & (n <= K)).all()
    t2, d2, x2, u2 = t.copy(), d.copy(), x.copy(), u.copy()
    for b in range(B):
        if n[b] < K:
            t2[b, n[b] + 1:] = rng.normal(0, 2, t2[b, n[b] + 1:].shape)
            d2[b, n[b] + 1:] = rng.normal(0, 2, d2[b, n[b] + 1:].shape)
            x2[b, n[b] + 1:] = rng.integers(0, V, K - n[b] - 1)
            u2[b, n[b] + 1:K] = rng.random(K - n[b] - 1)
    pert = oracle.verify_ref(t2, d2, x2, u2)
    np.testing.assert_array_equal(pert["accepted_len"], n)
    np.testing.assert_array_equal(pert["out_tokens"], base["out_tokens"])
    assert (n < K).sum() > 50


def test_identical_models_accept_everything_and_draw_the_bonus_from_p():
    rng = np.random.default_rng(6)
    B, K, V = 64, 5, 11
    t = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    d = t[:, :K].copy()
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    r = oracle.verify_ref(t, d, x, u)
    assert (r["accepted_len"] == K).all()
    np.testing.assert_array_equal(r["out_tokens"][:, :K], x)
    # V = 2 bonus row: token 0 iff u_K < p_K(0)
    t2 = np.zeros((2, 2, 2), np.float32)
    t2[:, 1] = [np.log(0.3), np.log(0.7)]
    r2 = oracle.verify_ref(t2, t2[:, :1].copy(), np.zeros((2, 1), np.int32),
                           np.array([[0.5, 0.2999], [0.5, 0.3001]], np.float32))
    assert list(r2["out_tokens"][:, 1]) == [0, 1]


def test_degenerate_shapes():
    # K = 0: the step is a single draw from p_0
    t = np.log(np.array([[[0.25, 0.75]]], np.float32))
    r = oracle.verify_ref(t, np.zeros((1, 0, 2), np.float32), np.zeros((1, 0), np.int32),
                          np.array([[0.2]], np.float32))
    assert r["accepted_len"][0] == 0 and list(r["out_tokens"][0]) == [0]
    # V = 1: p = q = 1, everything is accepted and the bonus is token 0
    t1 = np.zeros((3, 4, 1), np.float32)
    r = oracle.verify_ref(t1, t1[:, :3].copy(), np.zeros((3, 3), np.int32),
                          np.full((3, 4), 0.99, np.float32))
    assert (r["accepted_len"] == 3).all() and (r["out_tokens"] == 0).all()
    # B = 0
    r = oracle.verify_ref(np.zeros((0, 3, 5), np.float32), np.zeros((0, 2, 5), np.float32),
                          np.zeros((0, 2), np.int32), np.zeros((0, 3), np.float32))
    assert r["accepted_len"].shape == (0,)


def test_data_errors_are_reported_per_sequence():
    rng = np.random.default_rng(8)
    B, K, V = 4, 2, 6
    t = rng.normal(0, 1, (B, K + 1, V)).astype(np.float32)
    d = rng.normal(0, 1, (B, K, V)).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    x[1, 0] = V
    t[2, 2, 3] = np.nan
    u[3, 1] = 1.0
    r = oracle.verify_ref(t, d, x, u)
    assert r["status"] == oracle.DATA_TOKEN | oracle.DATA_LOGIT | oracle.DATA_UNIFORM
    assert r["accepted_len"][0] >= 0
    assert list(r["accepted_len"][1:]) == [-1, -1, -1]


def test_boundary_flags_mark_uniforms_near_a_threshold():
    t = [[0.0, 0.0], [0.0, 0.0]]
    d = [[np.log(3.0), 0.0]]
    r = _one(t, d, [0], [np.float32(2.0 / 3.0), 0.3])
    assert r["flags"][0] & oracle.FLAG_RATIO
    r = _one(t, d, [0], [0.2, 0.3])
    assert r["flags"][0] == 0
    # CDF boundary: accepted step, bonus row p = (0.5, 0.5), u_K at 0.5
    t2 = [[0.0, 0.0], [0.0, 0.0]]
    d2 = [[0.0, 0.0]]
    r = _one(t2, d2, [0], [0.1, 0.5])
    assert r["flags"][0] & oracle.FLAG_CDF


# --------------------------------------------------------------------------
# the drafter's sampling step (x ~ softmax(d / T) by inverse CDF)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_draft_sample_q_is_the_library_softmax_at_the_token(dtype):
    g = torch.Generator().manual_seed(11)
    x = torch.randn(6, 300, generator=g) * 3.0
    x[:, ::7] = float("-inf")
    u = torch.rand(6, generator=g)
    if dtype == "bf16":
        xb = x.to(torch.bfloat16)
        arr, xd = xb.view(torch.int16).numpy().view(np.uint16), xb.double()
    else:
        arr, xd = x.numpy(), x.double()
    r = oracle.draft_sample_ref(arr, u.numpy(), 0.8)
    p = torch.softmax(xd / 0.8, dim=-1).numpy()
    rows = np.arange(6)
    np.testing.assert_allclose(r["q_at"], p[rows, r["tokens"]], rtol=1e-12, atol=0)
    assert (p[rows, r["tokens"]] > 0).all()  # never a token without mass


def test_draft_sample_inverse_cdf_on_a_uniform_grid():
    """Uniforms on an even grid land in each token's CDF step in proportion to
    its probability: N*p_j of the N grid points, within one (plus float32
    rounding of the grid)."""
    logits = np.array([0.3, -1.2, 2.0, 0.0, -0.5], np.float32)
    N = 20000
    u = ((np.arange(N) + 0.5) / N).astype(np.float32)
    r = oracle.draft_sample_ref(np.tile(logits, (N, 1)), u, 1.0)
    p = torch.softmax(torch.tensor(logits, dtype=torch.float64), 0).numpy()
    counts = np.bincount(r["tokens"], minlength=5)
    assert np.abs(counts - N * p).max() <= 2.0
    # and the tokens are nondecreasing in u (an inverse CDF in token order)
    assert (np.diff(r["tokens"]) >= 0).all()


def test_draft_sample_equals_the_verifiers_bonus_draw():
    """With K = 0 the verifier's only draw is the bonus draw from p_0: the
    same inverse CDF on the same softmax."""
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(9, 1000, generator=g) * 4.0).numpy()
    u = torch.rand(9, generator=g).numpy()
    r = oracle.draft_sample_ref(x, u, 1.3)
    v = oracle.verify_ref(x[:, None, :], None, np.zeros((9, 0), np.int32), u[:, None], 1.3)
    np.testing.assert_array_equal(r["tokens"], v["out_tokens"][:, 0])


def test_draft_sample_data_errors():
    x = np.zeros((3, 10), np.float32)
    x[1, 4] = np.nan
    u = np.array([0.5, 0.5, 1.5], np.float32)
    r = oracle.draft_sample_ref(x, u, 1.0)
    assert r["status"] == oracle.DATA_LOGIT | oracle.DATA_UNIFORM


# --------------------------------------------------------------------------
# Speculative Rejection's cut ("Speculative Rejection" review, section 4.2,
# the speculative-rejection phase): r_cut is the alpha-quantile of the
# partial reward scores and the sequences scoring at least r_cut are kept.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("N", [1, 2, 7, 1000])
@pytest.mark.parametrize("alpha", [0.0, 0.1, 0.5, 0.731, 0.9, 1.0])
def test_rejection_cut_is_the_library_quantile(N, alpha):
    rng = np.random.default_rng(N * 31 + int(alpha * 1000))
    s = rng.standard_normal((32, N)).astype(np.float32)
    res = oracle.rejection_cut_ref(s, alpha)
    assert res["status"] == 0
    for g in range(s.shape[0]):
        row = s[g].astype(np.float64)
        q = np.quantile(row, alpha)  # linear interpolation between order statistics
        np.testing.assert_allclose(res["r_cut"][g], q, rtol=1e-12, atol=0)
        # no score sits within rounding of the cut, so the kept set is unique
        near = np.abs(row - q) <= 1e-9 * max(1.0, abs(q))
        exact_hits = row == res["r_cut"][g]
        assert not np.any(near & ~exact_hits)
        want = np.flatnonzero(row >= res["r_cut"][g])
        n = res["n_accepted"][g]
        assert n == want.size
        np.testing.assert_array_equal(res["accepted"][g, :n], want)
        assert np.all(res["accepted"][g, n:] == -1)


@pytest.mark.parametrize("N", [2, 5, 65, 1025])
def test_rejection_cut_on_the_order_statistic_grid(N):
    """alpha = k / (N - 1) puts the quantile exactly on the k-th smallest
    score; with distinct scores the cut keeps exactly N - k sequences.  N - 1
    is a power of two so that alpha * (N - 1) is exactly k in double."""
    rng = np.random.default_rng(N)
    perm = rng.permutation(N).astype(np.float32) * 0.5 - 7.0
    s = perm[None, :]
    for k in sorted({0, 1, N // 3, N // 2, N - 2, N - 1}):
        res = oracle.rejection_cut_ref(s, k / (N - 1))
        assert res["r_cut"][0] == k * 0.5 - 7.0
        assert res["n_accepted"][0] == N - k
        np.testing.assert_array_equal(res["accepted"][0, :N - k], np.flatnonzero(perm >= k * 0.5 - 7.0))


def test_rejection_cut_worked_by_hand():
    s = np.array([[3, 1, 4, 1, 5]], np.float32)  # sorted: 1 1 3 4 5
    cases = {0.5: (3.0, [0, 2, 4]),     # h = 2: the middle score, kept itself
             0.25: (1.0, [0, 1, 2, 3, 4]),  # h = 1: both ones tie with the cut
             0.6: (3.4, [2, 4]),        # h = 2.4: 3 + 0.4 * (4 - 3)
             1.0: (5.0, [4]),           # the best score alone
             0.0: (1.0, [0, 1, 2, 3, 4])}
    for alpha, (r, kept) in cases.items():
        res = oracle.rejection_cut_ref(s, alpha)
        assert res["r_cut"][0] == pytest.approx(r, rel=1e-15)
        n = res["n_accepted"][0]
        assert list(res["accepted"][0, :n]) == kept
        assert list(res["accepted"][0, n:]) == [-1] * (5 - n)


def test_rejection_cut_ties_keep_every_equal_score():
    s = np.full((3, 9), 2.5, np.float32)
    s[1, ::2] = -1.0  # 5 of -1, 4 of 2.5
    s[2] = np.array([0, 0, 1, 1, 1, 2, 2, 2, 2], np.float32)
    for alpha in [0.0, 0.3, 0.5, 0.99, 1.0]:
        res = oracle.rejection_cut_ref(s, alpha)
        assert res["n_accepted"][0] == 9
        for g in (1, 2):
            row = s[g].astype(np.float64)
            q = np.quantile(row, alpha)
            assert res["r_cut"][g] == pytest.approx(q, rel=1e-15, abs=1e-300)
            n = res["n_accepted"][g]
            np.testing.assert_array_equal(res["accepted"][g, :n], np.flatnonzero(row >= res["r_cut"][g]))


def test_rejection_cut_invariants():
    """More pruning never keeps more sequences; every kept score is at least
    every dropped one; the best sequence is always kept."""
    rng = np.random.default_rng(5)
    s = (rng.standard_normal((16, 257)) * 3).astype(np.float32)
    prev = None
    for alpha in np.linspace(0.0, 1.0, 21):
        res = oracle.rejection_cut_ref(s, alpha)
        n = res["n_accepted"]
        assert np.all(n >= 1)
        if prev is not None:
            assert np.all(n <= prev)
        prev = n
        for g in range(s.shape[0]):
            keep = res["accepted"][g, :n[g]]
            mask = np.zeros(s.shape[1], bool)
            mask[keep] = True
            assert np.argmax(s[g]) in keep
            if (~mask).any():
                assert s[g][mask].min() >= s[g][~mask].max()


def test_rejection_cut_data_errors_and_shapes():
    s = np.zeros((4, 6), np.float32)
    s[1, 3] = np.nan
    s[2, 0] = np.inf
    res = oracle.rejection_cut_ref(s, 0.5)
    assert res["status"] == oracle.DATA_SCORE
    assert list(res["n_accepted"]) == [6, 0, 0, 6]
    assert np.isnan(res["r_cut"][1]) and np.isnan(res["r_cut"][2])
    assert np.all(res["accepted"][1] == -1) and np.all(res["accepted"][2] == -1)
    for bad in (-0.1, 1.5, float("nan")):
        with pytest.raises(ValueError):
            oracle.rejection_cut_ref(s, bad)
    with pytest.raises(ValueError):
        oracle.rejection_cut_ref(np.zeros((2, 0), np.float32), 0.5)
    empty = oracle.rejection_cut_ref(np.zeros((0, 5), np.float32), 0.5)
    assert empty["status"] == 0 and empty["n_accepted"].size == 0


# --------------------------------------------------------------------------
# Speculative contrastive decoding ("논문 리뷰 [Speculative Contrastive
# Decoding]", section Speculative Contrastive Decoding): speculative sampling
# against the contrastive target P_n of expert and amateur, bonus from P_n.
# The page lost P_n's formula; the oracle reads it as contrastive decoding's
# log p_e - log p_a over the plausible head {p_e >= alpha max p_e}.  The
# pins below fix that reading to its verbal definition (library softmaxes,
# interior alpha, several temperatures), its two limits and the exactness of
# the verify step against it.
# --------------------------------------------------------------------------
def _scd_inputs(B, K, V, seed, T=1.0, amateur_zero=False):
    rng = np.random.default_rng(seed)
    t = (rng.standard_normal((B, K + 1, V)) * 3).astype(np.float32)
    t[:, :, 1] = -np.inf  # a masked token
    a = np.zeros_like(t) if amateur_zero else (t + rng.standard_normal(t.shape)).astype(np.float32)
    q = np.exp((a[:, :K] - a[:, :K].max(-1, keepdims=True)) / T)
    q /= q.sum(-1, keepdims=True)
    x = np.array([[rng.choice(V, p=q[b, i]) for i in range(K)] for b in range(B)], np.int32).reshape(B, K)
    u = rng.random((B, K + 1), dtype=np.float32)
    return t, a, x, u


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_scd_without_head_cut_and_a_flat_amateur_is_plain_speculative_sampling(T):
    """alpha = 0 keeps every finite token and a flat amateur shifts every
    contrast by a constant, so P_n = softmax(t / T) and q is uniform: the
    outputs are those of the plain verify with all-zero draft logits."""
    B, K, V = 64, 4, 50
    t, a, x, u = _scd_inputs(B, K, V, 3, T, amateur_zero=True)
    scd = oracle.scd_verify_ref(t, a, x, u, T, alpha=0.0, want_debug=True)
    plain = oracle.verify_ref(t, np.zeros((B, K, V), np.float32), x, u, T, want_debug=True)
    for k in ("accepted_len", "out_tokens", "p_at", "q_at", "flags"):
        np.testing.assert_array_equal(scd[k], plain[k], err_msg=k)
    assert scd["status"] == plain["status"] == 0


def test_scd_with_the_tightest_head_is_greedy_verification():
    """alpha = 1 leaves only the expert's argmax in the head, so P_n is a point
    mass there: every draft token that is not the argmax is rejected and
    replaced by it, which is Blockwise Parallel Decoding's greedy rule."""
    B, K, V = 200, 5, 40
    t, a, x, u = _scd_inputs(B, K, V, 4)
    g = t.argmax(-1)
    agree = np.random.default_rng(5).random((B, K)) < 0.6
    x = np.where(agree, g[:, :K], x).astype(np.int32)
    scd = oracle.scd_verify_ref(t, a, x, u, 1.0, alpha=1.0)
    greedy = oracle.verify_ref(t, None, x, None, mode=oracle.MODE_GREEDY)
    np.testing.assert_array_equal(scd["accepted_len"], greedy["accepted_len"])
    np.testing.assert_array_equal(scd["out_tokens"], greedy["out_tokens"])
    assert 0 < scd["accepted_len"].mean() < K


def test_scd_emitted_token_follows_the_contrastive_target():
    """The first emitted token is distributed as P_n at position 0, whatever
    the amateur proposes (the exactness of speculative sampling with target
    P_n); tokens outside the plausible head never appear."""
    V, K, T, alpha, n = 8, 2, 0.9, 0.2, 200000
    rng = np.random.default_rng(11)
    t1 = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    a1 = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    td, ad = t1.astype(np.float64), a1.astype(np.float64)
    head = td[0] >= td[0].max() + T * np.log(alpha)
    pn = np.where(head, np.exp((td[0] - ad[0]) / T), 0.0)
    pn /= pn.sum()
    assert 0 < (~head).sum() < V
    q = np.exp(ad[:K] / T)
    q /= q.sum(-1, keepdims=True)
    x = np.stack([rng.choice(V, size=n, p=q[i]) for i in range(K)], 1).astype(np.int32)
    u = rng.random((n, K + 1), dtype=np.float32)
    res = oracle.scd_verify_ref(np.broadcast_to(t1, (n, K + 1, V)), np.broadcast_to(a1, (n, K + 1, V)),
                                x, u, T, alpha)
    first = res["out_tokens"][:, 0]
    counts = np.bincount(first, minlength=V)
    assert counts[~head].sum() == 0
    _, pval = stats.chisquare(counts[head], n * pn[head])
    assert pval > 1e-3, pval
    # once x_0 is accepted, position 1 is a verify step of its own against
    # P_n at position 1 (accepted x_1 or the residual draw there)
    head1 = td[1] >= td[1].max() + T * np.log(alpha)
    pn1 = np.where(head1, np.exp((td[1] - ad[1]) / T), 0.0)
    pn1 /= pn1.sum()
    sel = res["accepted_len"] >= 1
    second = res["out_tokens"][sel, 1]
    counts1 = np.bincount(second, minlength=V)
    assert sel.sum() > 10000 and counts1[~head1].sum() == 0
    _, pval1 = stats.chisquare(counts1[head1], sel.sum() * pn1[head1])
    assert pval1 > 1e-3, pval1
    # with both accepted, the bonus token comes from P_n at position K = 2,
    # built from the expert's and the amateur's rows K
    head2 = td[2] >= td[2].max() + T * np.log(alpha)
    pn2 = np.where(head2, np.exp((td[2] - ad[2]) / T), 0.0)
    pn2 /= pn2.sum()
    sel2 = res["accepted_len"] == 2
    counts2 = np.bincount(res["out_tokens"][sel2, 2], minlength=V)
    assert sel2.sum() > 2000 and counts2[~head2].sum() == 0
    _, pval2 = stats.chisquare(counts2[head2], sel2.sum() * pn2[head2])
    assert pval2 > 1e-3, pval2


def _contrastive_by_definition(t_row, a_row, T, alpha):
    """P_n of one position built from its verbal definition with library
    softmaxes only: the plausible head is every token whose expert
    probability softmax(t/T) is at least alpha times the expert's largest
    probability, and P_n is the ratio expert / amateur of the two softmaxes
    (log p_e - log p_a) renormalised over that head, zero elsewhere.
    Returns (P_n, head, closest relative distance of a token to the cut)."""
    pe = torch.softmax(torch.from_numpy(t_row.astype(np.float64)) / T, 0)
    pa = torch.softmax(torch.from_numpy(a_row.astype(np.float64)) / T, 0)
    cut = alpha * pe.max()
    head = pe >= cut
    ratio = torch.where(head, pe / pa, torch.zeros_like(pe))
    pn = ratio / ratio.sum()
    gap = ((pe[pe > 0] - cut).abs() / cut).min().item()
    return pn.numpy(), head.numpy(), gap


@pytest.mark.parametrize("T,alpha", [(0.7, 0.1), (0.7, 0.5), (0.05, 0.3), (0.05, 0.8),
                                     (1.6, 0.25), (1.0, 0.05)])
def test_scd_contrastive_target_from_its_definition(T, alpha):
    """P_n away from both limits (0 < alpha < 1, T != 1), against the
    definition itself rather than the oracle's own threshold M + T ln(alpha):
    the oracle's P_n,i at EVERY token j (sequence j proposes x_i = j at each
    position i, so p_at[j, i] = P_n,i(j)) equals the renormalised ratio of
    two library softmaxes on the head {p_e >= alpha max p_e} to 1e-12, and is
    exactly zero off the head.  A head threshold without the temperature
    (M + ln alpha), a contrast without it (exp(t - a)) or an unrenormalised
    ratio would each fail here at these (T, alpha)."""
    V, K = 64, 3
    rng = np.random.default_rng(int(1000 * T + 100 * alpha))
    t = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    a = (t + rng.standard_normal((K + 1, V)) * 0.8).astype(np.float32)
    # a cluster of near-maximal logits in every row, so that the head at the
    # small temperatures holds several tokens (spacings 0.004-0.05 logits)
    for i in range(K + 1):
        top = t[i].max()
        idx = rng.choice(V, size=6, replace=False)
        t[i, idx] = top - np.cumsum(rng.uniform(0.004, 0.05, 6)).astype(np.float32)
    t[:, 7] = -np.inf  # a masked token: never in the head
    x = np.repeat(np.arange(V, dtype=np.int32)[:, None], K, 1)
    u = np.zeros((V, K + 1), np.float32)
    res = oracle.scd_verify_ref(np.broadcast_to(t, (V, K + 1, V)), np.broadcast_to(a, (V, K + 1, V)),
                                x, u, T, alpha, want_debug=True)
    assert res["status"] == 0
    sizes = []
    for i in range(K):
        pn, head, gap = _contrastive_by_definition(t[i], a[i], T, alpha)
        assert gap > 1e-9, "a token sits on the head's cut: the test would not decide it"
        got = res["p_at"][:, i]
        np.testing.assert_allclose(got, pn, rtol=1e-10, atol=1e-12, err_msg=f"position {i}")
        np.testing.assert_array_equal(got > 0, head, err_msg=f"support at position {i}")
        assert not head[7]
        sizes.append(int(head.sum()))
    # the cut is active and not trivial: neither every finite token nor only the argmax
    assert max(sizes) > 1 and min(sizes) < V - 1, sizes


def test_scd_contrastive_bonus_draw_from_its_definition():
    """The bonus token (all K accepted) comes from P_n at position K, the
    definition's law on rows K of expert and amateur: with uniforms on a
    grid, the emitted token is the inverse CDF of that law, pinned here as
    numpy's searchsorted on the cumulative definition (u away from steps)."""
    V, K, T, alpha = 24, 1, 0.7, 0.2
    rng = np.random.default_rng(77)
    t = (rng.standard_normal((K + 1, V)) * 1.2).astype(np.float32)
    a = (t + rng.standard_normal((K + 1, V)) * 0.7).astype(np.float32)
    pn0, head0, _ = _contrastive_by_definition(t[0], a[0], T, alpha)
    pnK, headK, gap = _contrastive_by_definition(t[K], a[K], T, alpha)
    assert gap > 1e-9 and 1 < headK.sum() < V
    # x_0 = the head token with the largest P_n,0 / q_0: accepted for every u
    qa = torch.softmax(torch.from_numpy(a[0].astype(np.float64)) / T, 0).numpy()
    x0 = int(np.argmax(np.where(head0, pn0 / qa, -1.0)))
    assert pn0[x0] >= qa[x0]
    cdf = np.cumsum(pnK)
    us = np.linspace(0.0, 0.999, 400).astype(np.float32)
    keep = np.min(np.abs(us[:, None].astype(np.float64) - cdf[None, :]), 1) > 1e-6
    us = us[keep]
    n = us.size
    u = np.zeros((n, K + 1), np.float32)
    u[:, K] = us
    res = oracle.scd_verify_ref(np.broadcast_to(t, (n, K + 1, V)), np.broadcast_to(a, (n, K + 1, V)),
                                np.full((n, K), x0, np.int32), u, T, alpha)
    assert np.all(res["accepted_len"] == K)
    want = np.searchsorted(cdf, us.astype(np.float64), side="right")
    np.testing.assert_array_equal(res["out_tokens"][:, K], want)
    assert set(np.unique(want)) == set(np.flatnonzero(headK))


def test_scd_data_errors_and_arguments():
    B, K, V = 4, 2, 16
    t, a, x, u = _scd_inputs(B, K, V, 6)
    a[1, 0, 5] = np.nan
    top = t[2, 1].argmax()
    a[2, 1, top] = -np.inf          # an unbounded contrast inside the head
    low = int(np.argsort(t[3, 0])[2])
    a[3, 0, low] = -np.inf          # outside the head (alpha = 0.5): harmless if t is low enough
    res = oracle.scd_verify_ref(t, a, x, u, 1.0, alpha=0.5)
    assert res["status"] == oracle.DATA_LOGIT
    assert res["accepted_len"][1] == -1 and res["accepted_len"][2] == -1
    assert res["accepted_len"][0] >= 0
    head3 = t[3, 0, low] >= t[3, 0].max() + np.log(0.5)
    assert (res["accepted_len"][3] >= 0) == (not head3)
    for bad in (-0.1, 1.5, float("nan")):
        with pytest.raises(ValueError):
            oracle.scd_verify_ref(t, a, x, u, 1.0, alpha=bad)


def test_rejection_cut_random_shapes_against_the_library_quantile():
    """Random prompt sizes, cut fractions and score patterns (ties, signed
    zeros, wide ranges) against numpy's linear quantile and the kept-set
    definition."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    @hyp.settings(max_examples=150, deadline=None)
    @hyp.given(st.integers(1, 300), st.floats(0.0, 1.0), st.integers(0, 2**31 - 1),
               st.sampled_from(["normal", "ties", "wide"]))
    def check(N, alpha, seed, kind):
        rng = np.random.default_rng(seed)
        if kind == "normal":
            s = rng.standard_normal((3, N))
        elif kind == "ties":
            s = rng.integers(-2, 3, (3, N)).astype(np.float64)
            s[s == 0] = np.where(rng.random((s == 0).sum()) < 0.5, -0.0, 0.0)
        else:
            s = rng.standard_normal((3, N)) * 10.0 ** rng.integers(-30, 30, (3, N))
        s = s.astype(np.float32)
        res = oracle.rejection_cut_ref(s, alpha)
        assert res["status"] == 0
        for g in range(3):
            row = s[g].astype(np.float64)
            q = np.quantile(row, alpha)
            assert res["r_cut"][g] == pytest.approx(q, rel=1e-12, abs=1e-300)
            n = res["n_accepted"][g]
            kept = res["accepted"][g, :n]
            np.testing.assert_array_equal(kept, np.flatnonzero(row >= res["r_cut"][g]))
            assert n >= 1 and np.all(res["accepted"][g, n:] == -1)

    check()
