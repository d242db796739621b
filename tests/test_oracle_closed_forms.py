"""Pins of the oracle's closed forms and elementwise helpers against the pages' printed numbers and
library routines."""
import math

import numpy as np
import pytest
import torch
from scipy.special import expit, logsumexp, softmax


def test_worked_example(orc, golden):
    g = golden("worked_example.json")
    words = orc.expected_words(g["alpha"], g["gamma"])
    assert abs(words - g["expected_words"]) < 0.005
    assert abs(words / (1 + g["gamma"] * g["c"]) - g["speedup"]) < 0.005
    assert abs(orc.speedup(g["alpha"], g["gamma"], g["c"]) - g["speedup"]) < 0.005
    assert abs(orc.speedup(0.4, 4, 0.1) - g["speedup_alpha_0_4"]) < 0.005


def test_worked_example_inconsistent_values_follow_formula(orc, golden):
    """Two printed sensitivities disagree with the page's own formula; the formula wins."""
    g = golden("worked_example.json")["printed_but_inconsistent"]
    s06 = orc.speedup(0.6, 4, 0.1)
    s8 = orc.speedup(0.8, 8, 0.1)
    assert abs(s06 - 1.6474) < 1e-3 and abs(s06 - g["speedup_alpha_0_6_printed"]) > 0.02
    assert abs(s8 - 2.4053) < 1e-3 and abs(s8 - g["speedup_gamma_8_printed"]) > 0.1


def test_expected_words_limits(orc):
    assert orc.expected_words(1.0, 7) == 8.0
    assert orc.expected_words(0.0, 7) == 1.0
    # geometric series 1 + a + ... + a^gamma, summed by brute force
    for a in (0.1, 0.5, 0.93):
        for gamma in (0, 1, 5, 16):
            assert abs(orc.expected_words(a, gamma) - sum(a**j for j in range(gamma + 1))) < 1e-12


def test_token_48_ratio(orc, golden):
    """p(48) = 0.007, q(48) = 0.025: the proposal is kept about 28% of the time."""
    g = golden("token_48.json")
    t = np.log([g["p"], 1 - g["p"]]).astype(np.float32)
    d = np.log([g["q"], 1 - g["q"]]).astype(np.float32)
    res, ratio = orc.verify_token_request(np.stack([t, t]), d[None], [0], seed=1, req=0)
    assert res.status == 0
    assert abs(ratio[0] - g["accept_probability"]) < 1e-6


def test_row_stats_match_logsumexp(orc):
    rng = np.random.default_rng(1)
    for V in (1, 7, 1000, 4097):
        row = (rng.normal(0, 4, V)).astype(np.float32)
        row[rng.integers(0, V, size=V // 10)] = -np.inf
        row[0] = 3.0
        st, M, S = orc.row_stats(row)
        assert st == 0
        assert M == row.max()
        assert abs(M + math.log(S) - logsumexp(row.astype(np.float64))) < 1e-12


def test_row_stats_errors(orc):
    assert orc.row_stats(np.array([1.0, np.nan], np.float32))[0] == orc.ERR_NAN
    assert orc.row_stats(np.array([1.0, np.inf], np.float32))[0] == orc.ERR_NAN
    assert orc.row_stats(np.array([-np.inf, -np.inf], np.float32))[0] == orc.ERR_NAN


def test_overlap_matches_library_softmax(orc):
    rng = np.random.default_rng(2)
    for V in (2, 16, 999):
        t = rng.normal(0, 2, V).astype(np.float32)
        d = (t + rng.normal(0, 1, V)).astype(np.float32)
        p, q = softmax(t.astype(np.float64)), softmax(d.astype(np.float64))
        assert abs(orc.overlap(t, d) - np.minimum(p, q).sum()) < 1e-12
        # identical rows overlap completely; min(p,q) + max(p-q,0) = p sums to one
        assert abs(orc.overlap(t, t) - 1.0) < 1e-12
        assert abs(np.minimum(p, q).sum() + np.maximum(p - q, 0).sum() - 1.0) < 1e-12


def _bf16_nearest_bruteforce(x):
    """Nearest bfloat16 to x by comparing bracketing bit patterns (ties to the even pattern)."""
    f = np.float32(x)
    base = int(np.array([f], np.float32).view(np.uint32)[0]) >> 16
    best = None
    for b in range(max(base - 3, 0), base + 4):
        if (b & 0x7F80) == 0x7F80:
            continue
        val = float(np.array([b << 16], np.uint32).view(np.float32)[0])
        if (x < 0) != (val < 0) and val != 0:
            continue
        key = (abs(val - x), b & 1)
        if best is None or key < best[0]:
            best = (key, b)
    return best[1]


def test_bf16_round_matches_library_and_bruteforce(orc):
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.normal(0, 3, 3000), rng.normal(0, 1e-3, 500),
                         np.ldexp(rng.uniform(1, 2, 200), rng.integers(-140, -120, 200)),
                         [0.0, 1.0, -2.5, 1.00390625, 1.01171875, 3.3e38]])
    for x in xs:
        got = orc.bf16_round(float(x))
        f32 = np.float32(x)
        if float(f32) == x:  # exactly a binary32: torch's single rounding is the library reference
            ref = torch.tensor([f32]).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
            assert got == ref, x
        if abs(x) > 1e-37:
            assert got == _bf16_nearest_bruteforce(float(x)) | (0x8000 if x < 0 else 0), x
    # a double halfway between two bfloat16 values that is not a binary32 halfway case
    x = 1.0 + 2**-8 + 2**-40  # just above the midpoint of 1 and 1 + 2^-7: rounds up
    assert orc.bf16_round(x) == 0x3F81
    assert orc.bf16_round(1.0 + 2**-8) == 0x3F80  # exact tie: even pattern
    assert orc.bf16_round(1.0 + 3 * 2**-8) == 0x3F82  # exact tie: even pattern


def test_sts_confidence_matches_expit(orc):
    rng = np.random.default_rng(4)
    for s, T in zip(rng.normal(0, 2, 50), rng.uniform(0.5, 1.5, 50)):
        assert abs(orc.sts_confidence(s, T) - expit(s / T)) < 1e-14
    assert orc.sts_confidence(0.0, 0.9) == 0.5
    # temperature scaling is monotone in the score: it never changes the ranking
    s = np.sort(rng.normal(0, 2, 20))
    c = [orc.sts_confidence(x, 1.3) for x in s]
    assert all(a < b for a, b in zip(c, c[1:]))


def test_lmhead_logits_pins(orc):
    """The output projection: a hand-worked 1 x 2 case, and random bf16-valued operands equal to
    a binary64 matrix product rounded once to binary32 (the operands' products are exact in
    binary64, so only the summation order differs: well inside one binary32 rounding)."""
    h = np.array([[1.0, 2.0, -0.5]], np.float32)
    W = np.array([[0.5, 0.25, 2.0], [-1.0, 1.0, 4.0]], np.float32)
    assert orc.lmhead_logits(h, W).tolist() == [[0.0, -1.0]]  # 0.5+0.5-1, -1+2-2
    import torch
    rng = np.random.default_rng(3)
    H = torch.from_numpy(rng.normal(0, 1, (5, 256)).astype(np.float32)).bfloat16().float().numpy()
    Wr = torch.from_numpy(rng.normal(0, 0.05, (300, 256)).astype(np.float32)).bfloat16().float()
    Wr = Wr.numpy()
    got = orc.lmhead_logits(H, Wr)
    ref = (H.astype(np.float64) @ Wr.astype(np.float64).T).astype(np.float32)
    assert np.abs(got.astype(np.float64) - ref).max() <= 2 * np.abs(ref).max() * 2.0 ** -24
