"""Pins of the oracle's adaptive-verification pieces ("How much does a token cost", "Adaptive
verification"): the scheduler's budget chosen as the best expected tokens per unit time over every
budget, and the per-position acceptance rates learned from what verification accepted."""
import numpy as np
import pytest

from speculative_decoding_verification_token_gb300 import synth


# ---- budget by the highest expected tokens per unit time ----------------------------------------

def _brute_force_argmax(c, max_len, sps, B_max):
    """Independent restatement in Python: float32 survival products, a tuple sort, exact integer
    fixed-point sums, and every budget evaluated."""
    N, K = c.shape
    items = []
    for i in range(N):
        S = np.float32(1.0)
        for k in range(1, int(max_len[i]) + 1):
            S = np.float32(S * np.float32(c[i, k - 1]))
            items.append((-float(S), k, i, float(S)))
    items.sort()
    b_lim = min(len(items), B_max - N)
    T = N << 40
    best, bstar = float(T) * 2.0 ** -40 * sps[N], 0
    for b in range(1, b_lim + 1):
        T += int(np.floor(items[b - 1][3] * 2.0 ** 40))
        f = float(T) * 2.0 ** -40 * sps[N + b]
        if f > best:
            best, bstar = f, b
    sel = np.zeros(N, np.int32)
    for _, _, i, _ in items[:bstar]:
        sel[i] += 1
    return sel, N + bstar, best


def test_argmax_hand_worked_two_peaks(orc):
    """One request, S = 0.5, 0.5.  f(0) = 1 * 1.0, f(1) = 1.5 * 0.6 = 0.9, f(2) = 2.0 * 0.6 = 1.2:
    the early stop keeps nothing (f(1) < f(0)); the best budget admits both drafts."""
    c = np.array([[0.5, 1.0]], np.float32)
    sps = np.array([0.0, 1.0, 0.6, 0.6])
    early = orc.schedule(c, [2], sps, 3, rule=orc.STOP_FIRST_DROP)
    best = orc.schedule(c, [2], sps, 3, rule=orc.STOP_ARGMAX)
    assert early["status"] == 0 and best["status"] == 0
    assert early["total_rows"] == 1 and list(early["sel_len"]) == [0]
    assert abs(early["objective"] - 1.0) < 1e-12
    assert best["total_rows"] == 3 and list(best["sel_len"]) == [2]
    assert abs(best["objective"] - 1.2) < 1e-12


def test_argmax_ties_take_the_smaller_budget(orc):
    """f(0) = 1, f(1) = 2 * 0.5 = 1: equal values keep the smaller budget."""
    c = np.array([[1.0]], np.float32)
    r = orc.schedule(c, [1], np.array([0.0, 1.0, 0.5]), 2, rule=orc.STOP_ARGMAX)
    assert r["total_rows"] == 1 and r["objective"] == 1.0


@pytest.mark.parametrize("seed", range(6))
def test_argmax_matches_brute_force(orc, seed):
    rng = np.random.default_rng(700 + seed)
    N, K = int(rng.integers(1, 9)), int(rng.integers(1, 7))
    c = rng.uniform(0.0, 1.0, (N, K)).astype(np.float32)
    c[rng.random((N, K)) < 0.1] = 1.0
    max_len = rng.integers(0, K + 1, N).astype(np.int32)
    B_max = int(N + rng.integers(0, N * K + 2))
    # a bumpy SPS curve, so that f has several local maxima
    sps = 1.0 / (1.0 + 0.05 * np.arange(B_max + 1)) * (1.0 + 0.3 * np.sin(np.arange(B_max + 1)))
    ref = _brute_force_argmax(c, max_len, sps, B_max)
    got = orc.schedule(c, max_len, sps, B_max, rule=orc.STOP_ARGMAX)
    assert got["status"] == 0
    assert (got["sel_len"] == ref[0]).all()
    assert got["total_rows"] == ref[1] and got["objective"] == ref[2]


@pytest.mark.parametrize("seed", range(4))
def test_argmax_dominates_early_stop(orc, seed):
    """The best budget's objective is never below the early stop's, and both admit a prefix of the
    same order (per request, the shorter prefixes first)."""
    rng = np.random.default_rng(800 + seed)
    N, K = 40, 8
    c = (rng.beta(8, 2, (N, K)) * 0.97 ** np.arange(K)).astype(np.float32)
    max_len = rng.integers(0, K + 1, N).astype(np.int32)
    B_max = N + 200
    sps = 1.0 / (2e-3 + np.arange(B_max + 1) * rng.uniform(1e-6, 3e-5))
    sps = sps * (1.0 + 0.02 * rng.standard_normal(B_max + 1))  # a noisy engine profile
    early = orc.schedule(c, max_len, sps, B_max, rule=orc.STOP_FIRST_DROP)
    best = orc.schedule(c, max_len, sps, B_max, rule=orc.STOP_ARGMAX)
    assert best["objective"] >= early["objective"]
    assert (best["sel_len"] <= max_len).all() and (early["sel_len"] <= max_len).all()
    assert best["total_rows"] == N + best["sel_len"].sum()


def test_argmax_equals_early_stop_when_f_is_log_concave(orc):
    """With a linear SPS curve, log f(b) = log T(b) + log SPS(N + b) is concave (T grows by
    non-increasing steps), so the first non-increase is the global maximum."""
    inp = synth.schedule_inputs(synth.SCHEDULE)
    N, B_max = inp["N"], inp["B_max"]
    sps = 500.0 - 0.05 * np.arange(B_max + 1)
    early = orc.schedule(inp["cond_accept"], inp["max_len"], sps, B_max, rule=orc.STOP_FIRST_DROP)
    best = orc.schedule(inp["cond_accept"], inp["max_len"], sps, B_max, rule=orc.STOP_ARGMAX)
    assert early["total_rows"] > N
    assert (early["sel_len"] == best["sel_len"]).all()
    assert early["objective"] == best["objective"]


# ---- per-position acceptance learned while serving ----------------------------------------------

def test_acceptance_hand_worked(orc):
    """Three requests, K = 4: verified (4, 2, 3), accepted (1, 2, 3).
    Reached: request 0 positions 1-2 (rejected at 2), request 1 positions 1-2 (all verified ones
    accepted), request 2 positions 1-3.  trials = (3, 3, 1, 0), accepts = (3, 2, 1, 0); with a
    Beta(1, 1) prior alpha = (4/5, 3/5, 2/3, 1/2)."""
    trials, accepts = np.zeros(4), np.zeros(4)
    st, alpha = orc.acceptance_update([4, 2, 3], [1, 2, 3], 4, trials, accepts)
    assert st == 0
    assert list(trials) == [3, 3, 1, 0] and list(accepts) == [3, 2, 1, 0]
    np.testing.assert_allclose(alpha, [0.8, 0.6, 2 / 3, 0.5], rtol=1e-7)


def test_acceptance_decay_closed_form(orc):
    """Two rounds with decay 1/2: trials = 1/2 * round 1 + round 2."""
    trials, accepts = np.zeros(3), np.zeros(3)
    orc.acceptance_update([3, 3], [3, 0], 3, trials, accepts, decay=0.5)   # (2,1,1) / (1,1,1)
    st, alpha = orc.acceptance_update([3], [1], 3, trials, accepts, decay=0.5,
                                      prior_a=2.0, prior_b=3.0)            # (1,1,0) / (1,0,0)
    assert st == 0
    np.testing.assert_array_equal(trials, [2.0, 1.5, 0.5])
    np.testing.assert_array_equal(accepts, [1.5, 0.5, 0.5])
    np.testing.assert_allclose(alpha, [(1.5 + 2) / (2 + 5), (0.5 + 2) / (1.5 + 5),
                                       (0.5 + 2) / (0.5 + 5)], rtol=1e-7)


def test_acceptance_converges_to_the_conditional_rates(orc):
    """Token-level verification of synthetic rounds where position k is accepted with probability
    a_k given that every earlier token was: the estimates converge to a_k (within four standard
    errors), for any verified lengths."""
    rng = np.random.default_rng(11)
    a = np.array([0.9, 0.75, 0.6, 0.5, 0.35])
    K = a.size
    trials, accepts = np.zeros(K), np.zeros(K)
    for _ in range(40):
        n = 5000
        sel = rng.integers(0, K + 1, n).astype(np.int32)
        ok = rng.random((n, K)) < a
        acc = np.where(ok.all(axis=1), K, np.argmin(ok, axis=1))  # first rejection
        acc = np.minimum(acc, sel).astype(np.int32)
        st, alpha = orc.acceptance_update(sel, acc, K, trials, accepts)
        assert st == 0
    se = np.sqrt(a * (1 - a) / trials)
    assert np.all(np.abs(alpha - a) < 4 * se), (alpha, a, se)
    # the counts can only shrink along the block: reaching k + 1 needs k accepted
    assert np.all(accepts <= trials) and np.all(trials[1:] <= accepts[:-1])


def test_acceptance_inconsistent_lengths(orc):
    trials, accepts = np.zeros(2), np.zeros(2)
    st, _ = orc.acceptance_update([1, 2], [2, 1], 2, trials, accepts)  # accepted > verified
    assert st != 0
    assert list(trials) == [1, 1] and list(accepts) == [1, 0]           # the bad request skipped


# ---- sequential temperature scaling ---------------------------------------------------------------

def _sequential_round(rng, N, K, Tstar, score_std=2.0, verified=None):
    """Confidence logits s and one verified round whose position-k outcome, given every earlier
    token accepted, is Bernoulli(sigma(s / Tstar_k))."""
    s = rng.normal(0.0, score_std, (N, K)).astype(np.float32)
    p = 1.0 / (1.0 + np.exp(-s.astype(np.float64) / np.asarray(Tstar)))
    ok = rng.random((N, K)) < p
    acc = np.where(ok.all(axis=1), K, np.argmin(ok, axis=1)).astype(np.int32)
    sel = np.full(N, K, np.int32) if verified is None else verified
    return s, sel, np.minimum(acc, sel).astype(np.int32)


def test_sts_recovers_known_temperatures(orc):
    """Outcomes drawn with temperatures (0.7, 1, 1.5, 2.5): each fitted T is within four standard
    errors of the true one (Fisher information of beta = 1 / T at the fit)."""
    rng = np.random.default_rng(21)
    Tstar = np.array([0.7, 1.0, 1.5, 2.5])
    s, sel, acc = _sequential_round(rng, 40000, 4, Tstar)
    r = orc.sts_fit(s, sel, acc)
    assert r["status"] == 0
    for k in range(4):
        reach = np.minimum(acc + 1, sel) >= k + 1
        x = s[reach, k].astype(np.float64)
        q = 1.0 / (1.0 + np.exp(-x / r["T"][k]))
        se_beta = 1.0 / np.sqrt(np.sum(q * (1 - q) * x * x))
        assert abs(1.0 / r["T"][k] - 1.0 / Tstar[k]) < 4 * se_beta, (k, r["T"][k], Tstar[k])
        assert r["count"][k] == reach.sum()
    assert np.all(r["ece_fit"][[0, 2, 3]] < r["ece_raw"][[0, 2, 3]])  # miscalibrated positions


def test_sts_matches_a_library_minimiser(orc):
    """The Newton fit equals scipy's bounded scalar minimisation of the same likelihood."""
    from scipy.optimize import minimize_scalar
    rng = np.random.default_rng(22)
    s, sel, acc = _sequential_round(rng, 3000, 3, [0.8, 1.3, 2.0],
                                    verified=rng.integers(0, 4, 3000).astype(np.int32))
    r = orc.sts_fit(s, sel, acc, iters=50)
    for k in range(3):
        reach = np.minimum(acc + 1, sel) >= k + 1
        x = s[reach, k].astype(np.float64)
        y = (acc[reach] >= k + 1).astype(np.float64)

        def nll(beta):
            z = -(2 * y - 1) * beta * x
            return np.sum(np.logaddexp(0.0, z))
        best = minimize_scalar(nll, bounds=(1 / 16, 16), method="bounded",
                               options={"xatol": 1e-10})
        assert abs(1.0 / r["T"][k] - best.x) < 1e-6 * best.x
        assert abs(r["nll"][k] - best.fun / reach.sum()) < 1e-9


def test_sts_calibrated_input_keeps_unit_temperature(orc):
    rng = np.random.default_rng(23)
    s, sel, acc = _sequential_round(rng, 60000, 2, [1.0, 1.0])
    r = orc.sts_fit(s, sel, acc)
    assert np.all(np.abs(r["T"] - 1.0) < 0.05)
    assert np.all(r["ece_raw"] < 0.02)


def test_sts_ece_hand_worked(orc):
    """Four samples at position 1 with confidences 1/4, 1/4, 3/4, 3/4 and labels 0, 1, 1, 1, two
    bins: |(0 - 1/4) + (1 - 1/4)| + |(1 - 3/4) + (1 - 3/4)| = 1, over 4 samples: 0.25."""
    s = np.array([[np.log(1 / 3)], [np.log(1 / 3)], [np.log(3)], [np.log(3)]], np.float32)
    sel = np.ones(4, np.int32)
    acc = np.array([0, 1, 1, 1], np.int32)
    r = orc.sts_fit(s, sel, acc, iters=0, nbins=2)
    assert r["T"][0] == 1.0 and r["count"][0] == 4
    assert abs(r["ece_raw"][0] - 0.25) < 1e-7 and r["ece_fit"][0] == r["ece_raw"][0]


def test_sts_preserves_the_order_of_confidences(orc):
    """Dividing by a positive temperature keeps every position's ranking of the scores."""
    rng = np.random.default_rng(24)
    s, sel, acc = _sequential_round(rng, 5000, 3, [0.5, 2.0, 4.0])
    T = orc.sts_fit(s, sel, acc)["T"]
    assert np.all(T > 0)
    for k in range(3):
        order = np.argsort(s[:, k], kind="stable")
        c = 1.0 / (1.0 + np.exp(-s[order, k].astype(np.float64) / float(T[k])))
        assert np.all(np.diff(c) >= 0.0)


# ---- fixed-depth cost model ---------------------------------------------------------------------

def test_fixed_depth_hand_worked(orc):
    """Two requests, c = (0.9, 0.5) and (0.5, 0.9): survivals (0.9, 0.45) and (0.5, 0.45).
    Depth 0, 1, 2: expected tokens L = 2, 3.4, 4.3 on B = 2, 4, 6 rows.  With step time
    C(B) = 1 + 0.1 B the throughput L / C is 1.67, 2.43, 2.69: depth 2.  With C(B) = 1 + 0.3 B it is
    1.25, 1.545, 1.536: slot 2 adds 0.9 expected tokens but would need 3.4 * (2.8 - 2.2) / 2.2 =
    0.93, so depth 1."""
    c = np.array([[0.9, 0.5], [0.5, 0.9]], np.float32)
    B = np.arange(7)
    r = orc.schedule(c, [2, 2], 1.0 / (1.0 + 0.1 * B), 6, rule=orc.STOP_FIXED_DEPTH)
    assert r["status"] == 0 and r["total_rows"] == 6 and list(r["sel_len"]) == [2, 2]
    assert abs(r["objective"] - 4.3 / 1.6) < 1e-6
    r = orc.schedule(c, [2, 2], 1.0 / (1.0 + 0.3 * B), 6, rule=orc.STOP_FIXED_DEPTH)
    assert r["total_rows"] == 4 and list(r["sel_len"]) == [1, 1]
    assert abs(r["objective"] - 3.4 / 2.2) < 1e-6


def _marginal_depth(c, max_len, sps, B_max):
    """The page's marginal rule in exact rational arithmetic: slot k + 1 pays while its survival
    mass p exceeds L_k (C_{k+1} - C_k) / C_k, with C = 1 / SPS."""
    from fractions import Fraction
    N, K = c.shape
    S = np.ones(N, np.float32)
    surv = []
    for k in range(1, K + 1):
        S = np.where(max_len >= k, (S * c[:, k - 1]).astype(np.float32), np.float32(0))
        surv.append([int(np.floor(float(s) * 2.0 ** 40)) if max_len[i] >= k else None
                     for i, s in enumerate(S)])
    L, B, depth = Fraction(N), N, 0
    for k in range(1, K + 1):
        add = [f for f in surv[k - 1] if f is not None]
        Bn = B + len(add)
        if Bn > B_max or Bn == B:
            break
        p = Fraction(sum(add), 2 ** 40)
        Ck, Cn = 1 / Fraction(sps[B]), 1 / Fraction(sps[Bn])
        if not p > L * (Cn - Ck) / Ck:
            break
        L, B, depth = L + p, Bn, k
    return depth, B


@pytest.mark.parametrize("seed", range(6))
def test_fixed_depth_is_the_marginal_rule(orc, seed):
    rng = np.random.default_rng(1300 + seed)
    N, K = int(rng.integers(1, 30)), int(rng.integers(1, 10))
    c = (rng.beta(8, 2, (N, K)) * 0.95 ** np.arange(K)).astype(np.float32)
    max_len = rng.integers(0, K + 1, N).astype(np.int32)
    B_max = int(N + rng.integers(0, N * K + 2))
    sps = 1.0 / (2e-3 + np.arange(B_max + 1) * rng.uniform(1e-5, 3e-4))
    depth, rows = _marginal_depth(c, max_len, sps, B_max)
    r = orc.schedule(c, max_len, sps, B_max, rule=orc.STOP_FIXED_DEPTH)
    assert r["status"] == 0
    assert r["total_rows"] == rows
    assert (r["sel_len"] == np.minimum(depth, max_len)).all()


@pytest.mark.parametrize("seed", range(4))
def test_best_budget_dominates_fixed_depth(orc, seed):
    """For any row count the sorted prefix holds the largest survivals, so the best budget over
    sorted prefixes is never below the fixed-depth choice."""
    rng = np.random.default_rng(1400 + seed)
    N, K = 50, 8
    c = (rng.beta(8, 2, (N, K)) * 0.97 ** np.arange(K)).astype(np.float32)
    max_len = rng.integers(0, K + 1, N).astype(np.int32)
    B_max = N * (K + 1)
    sps = 1.0 / (2e-3 + np.arange(B_max + 1) * 2e-5)
    best = orc.schedule(c, max_len, sps, B_max, rule=orc.STOP_ARGMAX)
    fixed = orc.schedule(c, max_len, sps, B_max, rule=orc.STOP_FIXED_DEPTH)
    assert best["objective"] >= fixed["objective"]


# ---- asynchronous scheduling: predictions from two rounds before -----------------------------

def test_schedule_async_three_rounds_by_hand(orc):
    """Two requests, one drafted position each, SPS = 1.0, 0.8, 0.7 at 2, 3, 4 verification rows.
    f(b) = (2 + first b survival values) * SPS(2 + b); admission stops at the first f(b + 1) <=
    f(b).  Rounds 0 and 1 have no two-rounds-old prediction and use the prior 0.3: f(1) = 2.3 *
    0.8 = 1.84 < 2 admits nothing.  Round 2 uses round 0's predictions (0.9, 0.6): f = 2, 2.32,
    3.5 * 0.7 = 2.45, both admitted.  Round 3 uses round 1's (0.2, 0.95): f = 2, 2.36, 2.205 --
    request 1 only.  Round 4 uses round 2's (0.1, 0.1): nothing."""
    prior = np.array([[0.3], [0.3]], np.float32)
    conf = np.array([[[0.9], [0.6]], [[0.2], [0.95]], [[0.1], [0.1]], [[0.99], [0.99]],
                     [[0.5], [0.5]]], np.float32)
    sps = np.array([1.0, 1.0, 1.0, 0.8, 0.7])
    want = {0: ([0, 0], 2), 1: ([0, 0], 2), 2: ([1, 1], 4), 3: ([0, 1], 3), 4: ([0, 0], 2)}
    for t, (sel, rows) in want.items():
        out = orc.schedule_async(conf, t, prior, [1, 1], sps, 4)
        assert out["status"] == 0
        assert list(out["sel_len"]) == sel and out["total_rows"] == rows, (t, out)
    assert orc.schedule_async(conf, 2, prior, [1, 1], sps, 4)["objective"] == pytest.approx(2.45)


def test_schedule_async_is_causal(orc):
    """Round t's selection does not depend on the predictions of rounds t and t - 1 (the tokens
    it admits), only on those of round t - 2."""
    rng = np.random.default_rng(17)
    N, K, T = 40, 6, 6
    conf = (rng.beta(8, 2, (T, N, K)) * 0.97 ** np.arange(K)).astype(np.float32)
    prior = np.full((N, K), 0.7, np.float32)
    ml = rng.integers(0, K + 1, N).astype(np.int32)
    sps = 1.0 / (2e-3 + np.arange(N * (K + 1) + 1) * 4e-6)
    for t in range(T):
        ref = orc.schedule_async(conf, t, prior, ml, sps, N * (K + 1))
        poked = conf.copy()
        poked[t] = 1.0 - poked[t]
        if t >= 1:
            poked[t - 1] = 0.0
        got = orc.schedule_async(poked, t, prior, ml, sps, N * (K + 1))
        assert (got["sel_len"] == ref["sel_len"]).all() and got["objective"] == ref["objective"]
        base = orc.schedule(conf[t - 2] if t >= 2 else prior, ml, sps, N * (K + 1))
        assert (base["sel_len"] == ref["sel_len"]).all()
