"""Helpers for the oracle's statistical pins: enumeration of every draft sequence on tiny vocabularies,
with Monte-Carlo over the verifier's own uniforms (distinct request ids give independent streams).

The target and draft distributions are the test's inputs (random logit tables indexed by the prefix),
so p(sequence) below is just the product of table entries: the definition of the target's joint
distribution, not a restatement of the verifier.
"""
import itertools

import numpy as np
from scipy.special import softmax


def prefix_tables(V, gamma, seed, target_std=1.5, draft_noise=1.0, context_free=False):
    """Logit tables T[prefix] (len <= gamma) and D[prefix] (len < gamma)."""
    rng = np.random.default_rng(seed)
    T, D = {}, {}
    base_t = rng.normal(0, target_std, V)
    base_d = base_t + rng.normal(0, draft_noise, V)
    for L in range(gamma + 1):
        for pre in itertools.product(range(V), repeat=L):
            if context_free:
                T[pre] = base_t.copy()
                if L < gamma:
                    D[pre] = base_d.copy()
            else:
                T[pre] = rng.normal(0, target_std, V)
                if L < gamma:
                    D[pre] = T[pre] + rng.normal(0, draft_noise, V)
    return T, D


def run_enumeration(orc, block, T, D, V, gamma, trials, seed, req_base=0):
    """For every draft sequence s: run `trials` verifications that differ only in the request id.

    Returns a list of (s, q(s), out) with out an int array [trials, gamma+1] (-1 padded)."""
    results = []
    req = req_base
    for s in itertools.product(range(V), repeat=gamma):
        qs = 1.0
        for i in range(gamma):
            qs *= softmax(D[s[:i]])[s[i]]
        t_rows = np.stack([T[s[:i]] for i in range(gamma + 1)]).astype(np.float32)
        d_rows = (np.stack([D[s[:i]] for i in range(gamma)]).astype(np.float32)
                  if gamma > 0 else np.zeros((1, V), np.float32))
        B = trials
        out = orc.verify_batch(
            block, t_rows, d_rows, V, V,
            target_row0=np.zeros(B, np.int64), draft_row0=np.zeros(B, np.int64),
            draft_len=np.full(B, gamma, np.int32),
            draft_tokens=np.array(s if gamma > 0 else [0], np.int32),
            B=B, seed=seed, request_ids=np.arange(req, req + B, dtype=np.uint64),
            out_ld=gamma + 1)
        assert out["status"] == 0
        req += B
        results.append((s, qs, out))
    return results


def p_joint(T, seq):
    pr = 1.0
    for j in range(len(seq)):
        pr *= softmax(T[tuple(seq[:j])])[seq[j]]
    return pr


def completion_zscores(T, V, gamma, results):
    """z-score, for every full sequence c of length gamma+1, of

        sum_tau P(emit c[:tau+1]) * p(c[tau+1:] | c[:tau+1])   versus   p(c).

    Emitting a prefix and then continuing from the target must reproduce the target's joint."""
    zs = []
    for c in itertools.product(range(V), repeat=gamma + 1):
        # coefficient of each possible emitted prefix length
        coef = np.zeros(gamma + 2)
        for tau in range(gamma + 1):
            rest = 1.0
            for j in range(tau + 1, gamma + 1):
                rest *= softmax(T[tuple(c[:j])])[c[j]]
            coef[tau] = rest
        est, var, n_min, q_max = 0.0, 0.0, None, 0.0
        for s, qs, out in results:
            toks = out["out_tokens"]
            tau = out["accepted_len"]
            n = toks.shape[0]
            x = np.zeros(n)
            for L in range(gamma + 1):
                sel = tau == L
                if not sel.any():
                    continue
                match = np.all(toks[sel, :L + 1] == np.array(c[:L + 1]), axis=1)
                x[np.flatnonzero(sel)[match]] = coef[L]
            est += qs * x.mean()
            var += qs * qs * x.var() / n
            n_min = n if n_min is None else min(n_min, n)
            q_max = max(q_max, qs)
        exact = p_joint(T, c)
        # X <= 1, so under the null sum_s q_s^2 E_s[X^2] / n <= q_max * p(c) / n: a floor for
        # cells too rare to be observed (their sample variance is zero)
        var = max(var, q_max * exact / n_min)
        zs.append((est - exact) / np.sqrt(var + 1e-300))
    return np.array(zs)


def mean_emitted(results):
    """Estimate of E[tau + 1] and its standard error over draft sequences weighted by q(s)."""
    est, var = 0.0, 0.0
    for s, qs, out in results:
        x = out["accepted_len"].astype(np.float64) + 1.0
        est += qs * x.mean()
        var += qs * qs * x.var() / x.size
    return est, np.sqrt(var)


def accept_first(results):
    """Estimate of P(tau >= 1) and its standard error."""
    est, var = 0.0, 0.0
    for s, qs, out in results:
        x = (out["accepted_len"] >= 1).astype(np.float64)
        est += qs * x.mean()
        var += qs * qs * x.var() / x.size
    return est, np.sqrt(var)
