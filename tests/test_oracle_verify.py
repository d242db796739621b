"""Pins of the oracle's token-level and block verification: losslessness by enumeration of every draft
sequence on tiny vocabularies, acceptance rate = sum min(p, q), expected words per round, the
block-verification toy, and the reduction of block to token verification at gamma = 1."""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

from mc_helpers import (accept_first, completion_zscores, mean_emitted, prefix_tables,
                        run_enumeration)


@pytest.mark.parametrize("block", [0, 1])
@pytest.mark.parametrize("V,gamma,trials", [(2, 2, 40000), (3, 2, 20000), (4, 3, 6000),
                                            (3, 3, 8000)])
def test_lossless_by_enumeration(orc, block, V, gamma, trials):
    """Emitting x_1..x_tau, Y and continuing from the target reproduces the target's joint
    distribution over every sequence of gamma+1 tokens (prefix-dependent random p, q tables)."""
    T, D = prefix_tables(V, gamma, seed=100 + 10 * V + gamma)
    res = run_enumeration(orc, block, T, D, V, gamma, trials, seed=9 + block)
    z = completion_zscores(T, V, gamma, res)
    assert np.abs(z).max() < 5.0, z


@pytest.mark.parametrize("block", [0, 1])
def test_first_token_follows_target(orc, block):
    """gamma = 1 on V = 16: the first emitted token is distributed as p_1."""
    V, gamma = 16, 1
    T, D = prefix_tables(V, gamma, seed=77, target_std=1.0, draft_noise=1.2)
    res = run_enumeration(orc, block, T, D, V, gamma, 20000, seed=3)
    p1 = softmax(T[()])
    for y in range(V):
        est, var = 0.0, 0.0
        for s, qs, out in res:
            x = (out["out_tokens"][:, 0] == y).astype(float)
            est += qs * x.mean()
            var += qs * qs * x.var() / x.size
        assert abs(est - p1[y]) < 5 * np.sqrt(var) + 1e-12


def test_accept_rate_is_overlap(orc):
    """P(first draft accepted) = sum_x min(p(x), q(x))."""
    V = 8
    T, D = prefix_tables(V, 1, seed=5)
    res = run_enumeration(orc, 0, T, D, V, 1, 30000, seed=4)
    est, se = accept_first(res)
    alpha = np.minimum(softmax(T[()]), softmax(D[()])).sum()
    assert abs(est - alpha) < 5 * se
    assert abs(orc.overlap(T[()].astype(np.float32), D[()].astype(np.float32)) - alpha) < 1e-6


def test_expected_words_empirical(orc):
    """Context-free p, q: mean emitted words per round = (1 - a^(gamma+1)) / (1 - a)."""
    V, gamma = 4, 4
    T, D = prefix_tables(V, gamma, seed=6, context_free=True)
    res = run_enumeration(orc, 0, T, D, V, gamma, 2000, seed=5)
    est, se = mean_emitted(res)
    alpha = np.minimum(softmax(T[()]), softmax(D[()])).sum()
    assert abs(est - orc.expected_words(alpha, gamma)) < 5 * se


def _toy_rows():
    p = np.log([1 / 3, 2 / 3])
    q = np.log([2 / 3, 1 / 3])
    return p.astype(np.float32), q.astype(np.float32)


def test_block_toy_running_ratio(orc, golden):
    g = golden("block_toy.json")
    t, d = _toy_rows()
    assert abs(softmax(t)[0] / softmax(d)[0] - g["ratio"]["A"]) < 1e-6
    assert abs(softmax(t)[1] / softmax(d)[1] - g["ratio"]["B"]) < 1e-6
    for name, toks in (("AB", [0, 1]), ("BA", [1, 0])):
        res, rho, h = orc.verify_block_request(np.stack([t, t, t]), np.stack([d, d]), toks, 1, 0)
        assert res.status == 0
        assert np.allclose(rho, g["running_ratio"][name], atol=1e-6)
    # AB: nothing spills past the first position (h_1 = 0) and the pair is kept whole (h_2 = 1)
    _, _, h = orc.verify_block_request(np.stack([t, t, t]), np.stack([d, d]), [0, 1], 1, 0)
    assert np.allclose(h, [0.0, 1.0], atol=1e-6)
    # BA: h_1 = 1, h_2 = rho_2 = 1/2
    _, _, h = orc.verify_block_request(np.stack([t, t, t]), np.stack([d, d]), [1, 0], 1, 0)
    assert np.allclose(h, [1.0, 0.5], atol=1e-6)


def test_block_toy_keeps_ab(orc, golden):
    """Draft AB is always kept whole by block verification; token-level keeps its A half the time."""
    g = golden("block_toy.json")
    t, d = _toy_rows()
    n = 4000
    kw = dict(target_row0=np.zeros(n, np.int64), draft_row0=np.zeros(n, np.int64),
              draft_len=np.full(n, 2, np.int32), draft_tokens=np.array([0, 1], np.int32), B=n,
              seed=11, request_ids=np.arange(n, dtype=np.uint64))
    blk = orc.verify_batch(1, np.stack([t, t, t]), np.stack([d, d]), 2, 2, **kw)
    tok = orc.verify_batch(0, np.stack([t, t, t]), np.stack([d, d]), 2, 2, **kw)
    assert (blk["accepted_len"] == 2).all()
    frac = (tok["accepted_len"] >= 1).mean()
    assert abs(frac - g["token_level_accepts_first_A"]) < 5 * np.sqrt(0.25 / n)
    # AB has the same probability 2/9 under the drafter and the target
    assert abs(softmax(d)[0] * softmax(d)[1] - g["prob_AB_under_q"]) < 1e-6
    assert abs(softmax(t)[0] * softmax(t)[1] - g["prob_AB_under_p"]) < 1e-6


def test_block_toy_output_distribution(orc, golden):
    """Toy, gamma = 2, drafts from q: emitted-and-completed pairs follow p x p (AB at 2/9)."""
    t, d = _toy_rows()
    T = {pre: t.astype(np.float64) for L in range(3) for pre in itertools.product(range(2), repeat=L)}
    D = {pre: d.astype(np.float64) for L in range(2) for pre in itertools.product(range(2), repeat=L)}
    res = run_enumeration(orc, 1, T, D, 2, 2, 30000, seed=12)
    z = completion_zscores(T, 2, 2, res)
    assert np.abs(z).max() < 5.0


def test_block_gamma1_equals_token(orc):
    """At gamma = 1 the block thresholds reduce to min(1, p/q) and the residual to max(p - q, 0):
    identical outputs for identical uniforms."""
    rng = np.random.default_rng(13)
    V, B = 50, 3000
    t = rng.normal(0, 2, (2, V)).astype(np.float32)
    d = (t[:1] + rng.normal(0, 1, (1, V))).astype(np.float32)
    st, toks = orc.sample_draft_batch(np.repeat(d, B, 0), V, V, np.arange(B), np.ones(B, np.int32),
                                      B, seed=21)
    assert st == 0
    kw = dict(target_row0=np.zeros(B, np.int64), draft_row0=np.arange(B, dtype=np.int64),
              draft_len=np.ones(B, np.int32), draft_tokens=toks, B=B, seed=22)
    a = orc.verify_batch(0, t, np.repeat(d, B, 0), V, V, **kw)
    b = orc.verify_batch(1, t, np.repeat(d, B, 0), V, V, **kw)
    assert (a["accepted_len"] == b["accepted_len"]).all()
    assert (a["out_tokens"] == b["out_tokens"]).all()
    assert np.allclose(a["ratio"], b["h"])


def test_block_accepts_at_least_as_much(orc):
    """Block verification's expected emitted length is never below token-level's."""
    V, gamma = 3, 3
    for seed in (31, 32):
        T, D = prefix_tables(V, gamma, seed=seed)
        tok = run_enumeration(orc, 0, T, D, V, gamma, 3000, seed=seed)
        blk = run_enumeration(orc, 1, T, D, V, gamma, 3000, seed=seed)
        (mt, st), (mb, sb) = mean_emitted(tok), mean_emitted(blk)
        assert mb > mt - 4 * np.hypot(st, sb)


def test_determinism_and_seed_dependence(orc):
    rng = np.random.default_rng(14)
    V, gamma, B = 300, 4, 64
    t = rng.normal(0, 3, (B * (gamma + 1), V)).astype(np.float32)
    d = (t.reshape(B, gamma + 1, V)[:, :gamma].reshape(-1, V)
         + rng.normal(0, 1, (B * gamma, V))).astype(np.float32)
    layout = dict(target_row0=np.arange(B) * (gamma + 1), draft_row0=np.arange(B) * gamma,
                  draft_len=np.full(B, gamma, np.int32), B=B)
    st, toks = orc.sample_draft_batch(d, V, V, layout["draft_row0"], layout["draft_len"], B, 5)
    for block in (0, 1):
        r1 = orc.verify_batch(block, t, d, V, V, draft_tokens=toks, seed=3, **layout)
        r2 = orc.verify_batch(block, t, d, V, V, draft_tokens=toks, seed=3, **layout)
        r3 = orc.verify_batch(block, t, d, V, V, draft_tokens=toks, seed=4, **layout)
        assert (r1["out_tokens"] == r2["out_tokens"]).all()
        assert not (r1["out_tokens"] == r3["out_tokens"]).all()


def test_edge_cases(orc):
    rng = np.random.default_rng(15)
    V = 20
    t = rng.normal(0, 1, (3, V)).astype(np.float32)
    d = (t[:2] + rng.normal(0, 1, (2, V))).astype(np.float32)
    # gamma = 0: only the bonus row is used
    res, _ = orc.verify_token_request(t[:1], d[:1], np.zeros(0, np.int32), 1, 0)
    assert res.status == 0 and res.accepted_len == 0 and res.race_kind == orc.RACE_BONUS
    # token ids outside [0, V)
    res, _ = orc.verify_token_request(t, d, [0, V], 1, 0)
    assert res.status == orc.ERR_TOKEN
    # q(x) = 0 for the drafted token is a data error
    d2 = d.copy()
    d2[0, 5] = -np.inf
    res, _ = orc.verify_token_request(t, d2, [5, 1], 1, 0)
    assert res.status == orc.ERR_ZERO_Q
    # NaN logits
    t2 = t.copy()
    t2[1, 3] = np.nan
    res, _ = orc.verify_token_request(t2, d, [0, 1], 1, 0)
    assert res.status == orc.ERR_NAN
    # masked (-inf) target entries are never emitted
    t3 = t.copy()
    t3[:, :10] = -np.inf
    for req in range(200):
        res, _ = orc.verify_token_request(t3, d, [15, 12], 7, req)
        assert res.status == 0 and res.correction >= 10


def test_identical_rows_accept_and_bonus(orc):
    """p = q: the ratio is exactly one, every draft is accepted (u < 1 always) and the emitted
    token after the draft is the bonus token, drawn from the target's next row."""
    V = 6
    t = np.log(np.full(V, 1.0 / V)).astype(np.float32)
    rows = np.stack([t, t])
    seen = set()
    for req in range(2000):
        res, ratio = orc.verify_token_request(rows, t[None], [2], 5, req)
        assert ratio[0] == 1.0
        assert res.accepted_len == 1 and res.race_kind == orc.RACE_BONUS
        seen.add(res.correction)
    assert seen == set(range(V))


def residual_empty_rows(V, x, seed):
    """One drafted position whose residual max(p - q, 0) is empty to working precision.

    The target masks token x (p(x) = 0) and the draft gives it the logit -120, a weight of
    about e^-120 of the row's scale; every other entry is the same in both rows.  So the ratio
    p(x)/q(x) is 0 (x is always rejected), and adding e^-120 to a normaliser of order one leaves it
    unchanged in binary64 and binary32 alike: p(y) = q(y) exactly for every y != x."""
    rng = np.random.default_rng(seed)
    t = rng.normal(0.0, 1.0, V).astype(np.float32)
    d = t.copy()
    t[x] = -np.inf
    d[x] = -120.0
    return t, d


@pytest.mark.parametrize("block", [0, 1])
def test_residual_empty_fallback(orc, block):
    """Rejection with an empty residual: the correction falls back to a race over p with the RESID
    uniforms of the rejected position, so the emitted token is distributed as p (chi-square over
    4000 requests), and x, which p excludes, never comes out."""
    from scipy.stats import chisquare
    V, x, n = 8, 5, 4000
    t, d = residual_empty_rows(V, x, seed=41)
    rows_t = np.stack([t, t])  # position 1 and the bonus row
    counts = np.zeros(V)
    for req in range(n):
        if block:
            res, rho, h = orc.verify_block_request(rows_t, d[None], [x], 7, req)
            assert rho[0] == 0.0 and h[0] == 0.0
        else:
            res, ratio = orc.verify_token_request(rows_t, d[None], [x], 7, req)
            assert ratio[0] == 0.0
        assert res.status == 0 and res.accepted_len == 0
        assert res.race_kind == orc.RACE_RESIDUAL_EMPTY
        counts[res.correction] += 1
    assert counts[x] == 0
    p = softmax(t.astype(np.float64))
    keep = p > 0
    stat = chisquare(counts[keep], n * p[keep] / p[keep].sum())
    assert stat.pvalue > 1e-4, (counts, n * p)


@pytest.mark.parametrize("block", [0, 1])
def test_emitted_histogram_chisquare_1e6(orc, block):
    """10^6 independent requests on V = 4, gamma = 2: drafts drawn from q by the oracle's sampler,
    verified; the first emitted token follows p_1 (chi-square, 3 degrees of freedom, the 1e-4
    critical value)."""
    from scipy.stats import chi2, chisquare
    V, G, n = 4, 2, 1_000_000
    rng = np.random.default_rng(2024)
    T = rng.normal(0, 1.0, (G + 1, V)).astype(np.float32)
    D = (T[:G] + rng.normal(0, 0.8, (G, V))).astype(np.float32)
    tgt, drf = np.tile(T, (n, 1)), np.tile(D, (n, 1))
    tr0 = np.arange(n, dtype=np.int64) * (G + 1)
    dr0 = np.arange(n, dtype=np.int64) * G
    dl = np.full(n, G, np.int32)
    st, toks = orc.sample_draft_batch(drf, V, V, dr0, dl, n, 11)
    assert st == 0
    out = orc.verify_batch(block, tgt, drf, V, V, tr0, dr0, dl, toks, n, 11, out_ld=G + 1)
    assert out["status"] == 0
    counts = np.bincount(out["out_tokens"][:, 0], minlength=V)
    stat = chisquare(counts, n * softmax(T[0].astype(np.float64))).statistic
    assert stat < chi2.ppf(1 - 1e-4, V - 1), (counts, stat)
