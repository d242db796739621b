"""GPU parity of dspark_sts_fit (sequential temperature scaling of the confidence head) with the
oracle: temperatures, losses, sample counts and calibration errors per position."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import build
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return sv


def _round(rng, N, K, Tstar, ragged):
    s = rng.normal(0.0, 2.0, (N, K)).astype(np.float32)
    p = 1.0 / (1.0 + np.exp(-s.astype(np.float64) / np.asarray(Tstar)))
    ok = rng.random((N, K)) < p
    acc = np.where(ok.all(axis=1), K, np.argmin(ok, axis=1)).astype(np.int32)
    sel = rng.integers(0, K + 1, N).astype(np.int32) if ragged else np.full(N, K, np.int32)
    return s, sel, np.minimum(acc, sel).astype(np.int32)


@pytest.mark.parametrize("N,K,ragged", [(32768, 16, False), (5000, 5, True), (2000, 3, True)])
def test_sts_fit_matches_oracle(sv, orc, N, K, ragged):
    rng = np.random.default_rng(N + K)
    Tstar = np.linspace(0.6, 2.4, K)
    s, sel, acc = _round(rng, N, K, Tstar, ragged)
    ref = orc.sts_fit(s, sel, acc)
    assert ref["status"] == 0
    out = sv.dspark_sts_fit(torch.from_numpy(s).cuda(), torch.from_numpy(sel).cuda(),
                            torch.from_numpy(acc).cuda())
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 0
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert (got["count"] == ref["count"]).all()
    # Positions with a well-posed fit (enough samples of both labels): the GPU evaluates the
    # logistic in binary32, so temperatures and losses agree to 1e-5 relative; a confidence within
    # 1e-6 of a bin edge may fall in the neighbouring bin, moving the calibration error by at most
    # 2 / n per such sample.  Positions reached by a handful of requests can have separable labels,
    # where the likelihood keeps improving as beta grows and both fits run toward the clamp at
    # different speeds: there the temperature need only lie inside the clamp.
    n = np.maximum(ref["count"], 1)
    pos = [(np.minimum(acc + 1, sel) >= k + 1) for k in range(K)]
    ones = np.array([np.sum(acc[m] >= k + 1) for k, m in enumerate(pos)])
    posed = (ref["count"] >= 100) & (ones >= 10) & (ref["count"] - ones >= 10)
    assert posed.sum() >= 2
    assert np.all(np.abs(got["T"] - ref["T"])[posed] <= 1e-5 * ref["T"][posed])
    assert np.all((np.abs(got["nll"] - ref["nll"]) <= 1e-5 * np.abs(ref["nll"]) + 1e-12)[posed])
    for key in ("ece_raw", "ece_fit"):
        tol = 1e-5 + 4.0 / n
        assert np.all((np.abs(got[key] - ref[key]) <= tol)[posed]), key
    assert np.all(np.abs(got["ece_raw"] - ref["ece_raw"]) <= 1e-5 + 4.0 / n)  # no fit involved
    assert np.all((got["T"] >= 1 / 16) & (got["T"] <= 16))


def test_sts_fit_reports_bad_lengths(sv):
    s = torch.zeros((2, 2), dtype=torch.float32, device="cuda")
    out = sv.dspark_sts_fit(s, torch.tensor([1, 2], dtype=torch.int32, device="cuda"),
                            torch.tensor([2, 0], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(out["status"].item()) == sv.SV_ERR_BAD_INPUT
