"""GPU parity of dspark_schedule with the oracle (bit-exact selections), and the scheduled round:
the scheduler's lengths feed token-level verification without a host round trip."""
import numpy as np
import pytest
import torch

from parity import compare_verify, layout_np, oracle_tokens, oracle_verify
from speculative_decoding_verification_token_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import build
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return sv


def _gpu_schedule(sv, c, max_len, sps, B_max):
    out = sv.dspark_schedule(torch.from_numpy(np.ascontiguousarray(c)).cuda(),
                             torch.from_numpy(np.ascontiguousarray(max_len, np.int32)).cuda(),
                             torch.from_numpy(np.ascontiguousarray(sps, np.float64)).cuda(), B_max)
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


def _check(sv, orc, c, max_len, sps, B_max):
    ref = orc.schedule(c, max_len, sps, B_max)
    assert ref["status"] == 0
    got = _gpu_schedule(sv, c, max_len, sps, B_max)
    assert (got["sel_len"] == ref["sel_len"]).all()
    assert int(got["total_rows"][0]) == ref["total_rows"]
    assert got["objective"][0] == ref["objective"]
    assert (got["survival"].view(np.uint32) == ref["survival"].view(np.uint32)).all()
    return got


def test_schedule_512_request_workload(sv, orc):
    inp = synth.schedule_inputs(synth.SCHEDULE)
    got = _check(sv, orc, inp["cond_accept"], inp["max_len"], inp["sps"], inp["B_max"])
    assert 4.0 <= got["total_rows"][0] / inp["N"] <= 6.5


@pytest.mark.parametrize("seed", range(8))
def test_schedule_random_with_ties(sv, orc, seed):
    rng = np.random.default_rng(200 + seed)
    N = int(rng.integers(1, 700))
    K = int(rng.integers(1, 20))
    if N * K > 16384:
        N = 16384 // K
    c = (rng.beta(8, 2, (N, K)) * 0.97 ** np.arange(K)).astype(np.float32)
    c[rng.random((N, K)) < 0.05] = 1.0
    c[rng.random((N, K)) < 0.02] = 0.0
    if N > 2:
        c[1::3] = c[0:N - 1:3][: len(c[1::3])]
    max_len = rng.integers(0, K + 1, N).astype(np.int32)
    B_max = int(N + rng.integers(0, 3 * N * K // 4 + 2))
    per_row = rng.uniform(1e-8, 1e-4)
    sps = 1.0 / (2e-3 + np.arange(B_max + 1) * per_row)
    _check(sv, orc, c, max_len, sps, B_max)


def test_schedule_edge_cases(sv, orc):
    c = np.array([[0.95, 0.95, 0.95, 0.95]], np.float32)
    _check(sv, orc, c, [4], np.array([1.0, 1.0, 0.4, 0.9, 0.9, 0.9]), 5)  # early stop at 0
    c3 = np.array([[0.9, 0.5]] * 3, np.float32)
    _check(sv, orc, c3, [2, 2, 2], np.ones(5), 4)                         # ties -> request 0
    _check(sv, orc, c3, [0, 0, 0], np.ones(5), 4)                         # nothing extendable
    big = np.full((128, 128), 0.999, np.float32)
    _check(sv, orc, big, np.full(128, 128, np.int32), 1.0 / (1 + 1e-4 * np.arange(16385)),
           16384)                                                         # 16384 items


def test_scheduled_round(sv, orc):
    """Schedule 64 requests x 16 positions, then verify exactly the selected prefixes."""
    N, K = 64, 16
    sw = synth.ScheduleWorkload("sched64", N, K, 2048, 2.0, 0.4, 0.97, 8.0, 2.0, 7)
    si = synth.schedule_inputs(sw)
    vw = synth.scaled(synth.SCHEDULED_VERIFY, B=N, gamma=K, V=30000)
    vin = synth.token_inputs(vw, device="cpu")
    tokens = oracle_tokens(orc, vin)  # all 16 drafted tokens of every request
    # device chain: scheduler lengths go straight into the verifier
    sched = sv.dspark_schedule(torch.from_numpy(si["cond_accept"]).cuda(),
                               torch.from_numpy(si["max_len"]).cuda(),
                               torch.from_numpy(si["sps"]).cuda(), si["B_max"])
    d = dict(vin)
    for k in ("target", "draft", "target_row0", "draft_row0"):
        d[k] = vin[k].cuda()
    d["draft_len"] = sched["sel_len"]
    gpu = sv.spec_verify_token(d["target"], d["draft"], d["target_row0"], d["draft_row0"],
                               d["draft_len"], K, torch.from_numpy(tokens).cuda(), d["seed"])
    torch.cuda.synchronize()
    assert int(gpu["status"].item()) == 0
    ref_s = orc.schedule(si["cond_accept"], si["max_len"], si["sps"], si["B_max"])
    assert (sched["sel_len"].cpu().numpy() == ref_s["sel_len"]).all()
    vin["draft_len"] = torch.from_numpy(ref_s["sel_len"])
    ref = oracle_verify(orc, 0, vin, tokens)
    lay = layout_np(vin)
    res = compare_verify(gpu, ref, 0, lay["draft_len"], lay["draft_row0"])
    print(f"\n[parity] scheduled round: {res}")
