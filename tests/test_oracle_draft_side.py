"""Pins of the oracle's DSpark draft side: Markov-head drafting (special cases, brute-force product,
sampling statistics) and the confidence scheduler (hand-worked example, naive re-evaluation, early
stop, load response, plausibility on the 512-request workload)."""
import numpy as np
import pytest
import torch
from scipy.special import expit, logsumexp, softmax

from speculative_decoding_verification_token_gb300 import synth


def _bf16_vals(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_of_f32(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().astype(np.uint16)


def _nearest_bf16_bits(x):
    """Brute force: nearest bfloat16 pattern to each double (ties to the even pattern)."""
    x = np.asarray(x, np.float64)
    base = (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.int64)
    best = np.zeros(x.shape, np.int64)
    bestd = np.full(x.shape, np.inf)
    for off in range(-2, 3):
        cand = np.clip(base + off, 0, 0xFFFF)
        vals = _bf16_vals(cand)
        d = np.abs(vals - x)
        better = (d < bestd) | ((d == bestd) & ((cand & 1) == 0))
        best = np.where(better, cand, best)
        bestd = np.where(better, d, bestd)
    return best.astype(np.uint16)


def _markov_case(rng, K=4, V=8, R=3, wstd=0.7, bstd=1.5):
    backbone = rng.normal(0, bstd, (K, V)).astype(np.float32)
    U = rng.normal(0, wstd, (V, R)).astype(np.float32)
    W = rng.normal(0, wstd, (R, V)).astype(np.float32)
    scores = rng.normal(0, 1, K).astype(np.float32)
    T = rng.uniform(0.8, 1.2, K).astype(np.float32)
    return backbone, U, W, scores, T


def test_markov_bruteforce_product():
    """V <= 8: z_k = nearest-bf16(backbone_k + U[x_{k-1}] @ W) with the product in float64."""
    import oracle
    rng = np.random.default_rng(40)
    for trial in range(20):
        backbone, U, W, scores, T = _markov_case(rng)
        anchor = int(rng.integers(0, 8))
        out = oracle.markov_draft_request(backbone, U, W, anchor, scores, T, seed=3, req=trial)
        assert out["status"] == 0
        prev = anchor
        for k in range(backbone.shape[0]):
            exact = backbone[k].astype(np.float64) + U[prev].astype(np.float64) @ W.astype(np.float64)
            assert (out["z"][k] == _nearest_bf16_bits(exact)).all()
            z = _bf16_vals(out["z"][k])
            assert out["stats"][k, 0] == z.max()
            assert abs(out["stats"][k, 1] - logsumexp(z)) < 1e-12
            assert abs(out["conf"][k] - expit(np.float64(scores[k]) / np.float64(T[k]))) < 1e-12
            prev = out["x"][k]


def test_markov_zero_transition_is_plain_sampling():
    """U = 0: z is the bf16-rounded backbone and x_k its exponential-race sample (DRAFT tag, pos k)."""
    import oracle
    rng = np.random.default_rng(41)
    backbone, U, W, scores, T = _markov_case(rng, K=5, V=64, R=16)
    U[:] = 0
    out = oracle.markov_draft_request(backbone, U, W, 7, scores, T, seed=9, req=4)
    assert (out["z"] == _bf16_of_f32(backbone)).all()
    for k in range(5):
        st, tok, _ = oracle.sample_race(_bf16_vals(out["z"][k]).astype(np.float32), 9, 4, k + 1,
                                        oracle.TAG_DRAFT)
        assert tok == out["x"][k]


def test_markov_forced_transitions():
    """A one-hot transition table that dwarfs the backbone forces x_k = f(x_{k-1})."""
    import oracle
    V, R, K = 32, 32, 8
    perm = np.random.default_rng(42).permutation(V)
    backbone = np.zeros((K, V), np.float32)
    U = np.eye(V, R, dtype=np.float32) * 64.0          # U[x] = 64 e_x
    W = np.zeros((R, V), np.float32)
    W[np.arange(R), perm] = 1.0                        # e_j . W = e_{perm[j]}
    out = oracle.markov_draft_request(backbone, U, W, 5, np.zeros(K, np.float32),
                                      np.ones(K, np.float32), seed=1, req=0)
    x, prev = [], 5
    for _ in range(K):
        prev = perm[prev]
        x.append(prev)
    assert out["x"].tolist() == x


def test_markov_teacher_forcing():
    import oracle
    rng = np.random.default_rng(43)
    backbone, U, W, scores, T = _markov_case(rng, K=4, V=8, R=3)
    forced = np.array([1, 6, 2, 0], np.int32)
    out = oracle.markov_draft_request(backbone, U, W, 3, scores, T, 2, 0, forced_prev=forced)
    for k in range(4):
        exact = backbone[k].astype(np.float64) + U[forced[k]].astype(np.float64) @ W
        assert (out["z"][k] == _nearest_bf16_bits(exact)).all()


def test_markov_first_sample_follows_softmax():
    """Chi-square: x_1 over many request ids is distributed as softmax(z_1)."""
    import oracle
    rng = np.random.default_rng(44)
    backbone, U, W, scores, T = _markov_case(rng, K=1, V=8, R=3, bstd=0.8)
    n = 20000
    counts = np.zeros(8)
    z1 = None
    for req in range(n):
        out = oracle.markov_draft_request(backbone, U, W, 2, scores, T, seed=17, req=req,
                                          want_z=(req == 0))
        if z1 is None:
            z1 = _bf16_vals(out["z"][0])
        counts[out["x"][0]] += 1
    expct = softmax(z1) * n
    chi2 = ((counts - expct) ** 2 / expct).sum()
    assert chi2 < 30  # 7 degrees of freedom; p ~ 1e-4 at 30


# ---- scheduler ----------------------------------------------------------------------------

def test_schedule_hand_worked():
    """Two requests, three positions each; c = [[.9,.8,.5],[.6,.5,.9]] gives survival
    [.9,.72,.36] and [.6,.3,.27]; in order .9,.72,.6,.36,.3,.27 the expected-accepted totals are
    2, 2.9, 3.62, 4.22, 4.58, 4.88, 5.15 (one guaranteed token per request).
    SPS(B) = 1/(1 + 0.1 B):  f = 1.667, 2.231, 2.586, 2.813, 2.863, 2.871, 2.861 -> stop at b = 5:
    request 0 keeps 3 drafts, request 1 keeps 2, 7 verification rows.
    SPS(B) = 1/(1 + 0.5 B):  f = 1.0, 1.16, 1.207, 1.206 -> stop at b = 2: lengths [2, 0]."""
    import oracle
    c = np.array([[0.9, 0.8, 0.5], [0.6, 0.5, 0.9]], np.float32)
    Bs = np.arange(11)
    r = oracle.schedule(c, [3, 3], 1.0 / (1 + 0.1 * Bs), 10)
    assert r["status"] == 0
    assert r["sel_len"].tolist() == [3, 2] and r["total_rows"] == 7
    assert abs(r["objective"] - 4.88 / 1.7) < 1e-6
    assert np.allclose(r["survival"], [[0.9, 0.72, 0.36], [0.6, 0.3, 0.27]], atol=1e-6)
    r = oracle.schedule(c, [3, 3], 1.0 / (1 + 0.5 * Bs), 10)
    assert r["sel_len"].tolist() == [2, 0] and r["total_rows"] == 4
    # the row budget caps admission: B_max = 4 allows two drafts only
    r = oracle.schedule(c, [3, 3], 1.0 / (1 + 0.1 * Bs[:5]), 4)
    assert r["sel_len"].tolist() == [2, 0] and r["total_rows"] == 4


def _naive_frontier_schedule(c, max_len, sps, B_max):
    """O(n^2) re-evaluation: each step scans every request's next unadmitted position, admits the
    most probable one, recomputes the objective from scratch, and stops at the first step that
    does not raise it."""
    N, K = c.shape
    surv = np.zeros((N, K), np.float32)
    for i in range(N):
        s = np.float32(1.0)
        for k in range(max_len[i]):
            s = np.float32(s * c[i, k])
            surv[i, k] = s
    sel = [0] * N

    def objective(sel):
        tot = N * (1 << 40) + sum(int(np.floor(np.float64(surv[i, k]) * 2.0**40))
                                  for i in range(N) for k in range(sel[i]))
        return float(tot) * 2.0**-40 * sps[N + sum(sel)]

    f = objective(sel)
    while N + sum(sel) + 1 <= B_max:
        cands = [(-float(surv[i, sel[i]]), sel[i] + 1, i) for i in range(N) if sel[i] < max_len[i]]
        if not cands:
            break
        _, _, i = min(cands)
        sel[i] += 1
        fn = objective(sel)
        if not fn > f:
            sel[i] -= 1
            break
        f = fn
    return sel, f


@pytest.mark.parametrize("seed", range(6))
def test_schedule_matches_naive_reevaluation(seed):
    import oracle
    rng = np.random.default_rng(50 + seed)
    N, K = 24, 7
    c = (rng.beta(8, 2, (N, K)) * 0.97 ** np.arange(K)).astype(np.float32)
    if seed % 2:
        c[rng.random((N, K)) < 0.1] = 1.0  # survival repeats along a request
        c[1::2] = c[0::2]                  # identical requests: ties broken by request index
    max_len = rng.integers(0, K + 1, N).astype(np.int32)
    B_max = 120
    sps = 1.0 / (2e-3 + np.arange(B_max + 1) * rng.uniform(2e-5, 2e-4))
    r = oracle.schedule(c, max_len, sps, B_max)
    sel, f = _naive_frontier_schedule(c, max_len, sps, B_max)
    assert r["sel_len"].tolist() == sel
    assert r["objective"] == f
    assert r["total_rows"] == N + sum(sel)


def test_schedule_early_stop_does_not_look_ahead():
    """An engine curve with a dip: f falls at b = 1 and rises again later.  The scheduler stops at
    the first non-increase instead of taking the best budget over all b."""
    import oracle
    c = np.array([[0.95, 0.95, 0.95, 0.95]], np.float32)
    sps = np.array([1.0, 1.0, 0.4, 0.9, 0.9, 0.9])
    r = oracle.schedule(c, [4], sps, 5)
    assert r["sel_len"].tolist() == [0] and r["total_rows"] == 1
    best_b = int(np.argmax([(1 + np.cumprod(c[0])[:b].sum()) * sps[1 + b] for b in range(5)]))
    assert best_b > 0  # a look-ahead search would have admitted drafts


def test_schedule_tightens_under_load():
    import oracle
    inp = synth.schedule_inputs(synth.SCHEDULE)
    c, ml = inp["cond_accept"][:64], inp["max_len"][:64]
    prev = None
    for per_row in (0.05e-6, 0.4e-6, 4e-6, 40e-6, 400e-6):
        sps = 1.0 / (2e-3 + np.arange(8193) * per_row)
        r = oracle.schedule(c, ml, sps, 8192)
        tot = int(r["sel_len"].sum())
        if prev is not None:
            assert tot <= prev
        prev = tot
    assert prev < 64  # a heavily loaded engine keeps only the safest bets


def test_schedule_plausible_on_512_request_workload():
    """Light load on the synthetic curve verifies about 4-6 tokens per request."""
    import oracle
    inp = synth.schedule_inputs(synth.SCHEDULE)
    r = oracle.schedule(inp["cond_accept"], inp["max_len"], inp["sps"], inp["B_max"])
    assert r["status"] == 0
    per_request = r["total_rows"] / inp["N"]
    assert 4.0 <= per_request <= 6.5
    assert (r["sel_len"] <= inp["max_len"]).all()


def test_schedule_errors():
    import oracle
    c = np.array([[0.5, np.nan]], np.float32)
    assert oracle.schedule(c, [2], np.ones(5), 4)["status"] == oracle.ERR_NAN
    assert oracle.schedule(np.ones((3, 2), np.float32) * .5, [2, 2, 2], np.ones(5), 2)["status"] == oracle.ERR_ARGS


def test_schedule_ties_go_to_lower_request():
    """Equal survival: the lower request index is admitted first (row budget allows one draft)."""
    import oracle
    c = np.array([[0.9, 0.5], [0.9, 0.5], [0.9, 0.5]], np.float32)
    r = oracle.schedule(c, [2, 2, 2], np.ones(5), 4)
    assert r["sel_len"].tolist() == [1, 0, 0]
    r = oracle.schedule(c, [2, 2, 2], np.ones(6), 5)
    assert r["sel_len"].tolist() == [1, 1, 0]
