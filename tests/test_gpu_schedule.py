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


# ---- adaptive verification: best-budget rule and learned per-position acceptance ---------------

def _gpu_schedule_rule(sv, c, max_len, sps, B_max, rule):
    out = sv.dspark_schedule(torch.from_numpy(np.ascontiguousarray(c)).cuda(),
                             torch.from_numpy(np.ascontiguousarray(max_len, np.int32)).cuda(),
                             torch.from_numpy(np.ascontiguousarray(sps, np.float64)).cuda(), B_max,
                             rule=rule)
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("rule", ["argmax", "fixed_depth"])
@pytest.mark.parametrize("seed", range(6))
def test_schedule_argmax_rule_matches_oracle(sv, orc, seed, rule):
    """Best budget over all budgets, and one depth for every request, bit-exact, on random tables
    with a bumpy SPS curve (several local maxima of f) and ties."""
    rng = np.random.default_rng(900 + seed)
    N = int(rng.integers(1, 700))
    K = int(rng.integers(1, 20))
    if N * K > 16384:
        N = 16384 // K
    c = (rng.beta(8, 2, (N, K)) * 0.97 ** np.arange(K)).astype(np.float32)
    c[rng.random((N, K)) < 0.05] = 1.0
    if N > 2:
        c[1::3] = c[0:N - 1:3][: len(c[1::3])]
    max_len = rng.integers(0, K + 1, N).astype(np.int32)
    B_max = int(N + rng.integers(0, 3 * N * K // 4 + 2))
    b = np.arange(B_max + 1)
    sps = 1.0 / (2e-3 + b * rng.uniform(1e-8, 1e-4)) * (1.0 + 0.05 * np.sin(0.3 * b))
    o_rule, g_rule = ((orc.STOP_ARGMAX, sv.SV_STOP_ARGMAX) if rule == "argmax"
                      else (orc.STOP_FIXED_DEPTH, sv.SV_STOP_FIXED_DEPTH))
    ref = orc.schedule(c, max_len, sps, B_max, rule=o_rule)
    assert ref["status"] == 0
    got = _gpu_schedule_rule(sv, c, max_len, sps, B_max, g_rule)
    assert (got["sel_len"] == ref["sel_len"]).all()
    assert int(got["total_rows"][0]) == ref["total_rows"]
    assert got["objective"][0] == ref["objective"]


def test_schedule_argmax_rule_workload_and_edges(sv, orc):
    inp = synth.schedule_inputs(synth.SCHEDULE)
    for rule in (sv.SV_STOP_ARGMAX, sv.SV_STOP_FIRST_DROP, sv.SV_STOP_FIXED_DEPTH):
        ref = orc.schedule(inp["cond_accept"], inp["max_len"], inp["sps"], inp["B_max"],
                           rule=rule)
        got = _gpu_schedule_rule(sv, inp["cond_accept"], inp["max_len"], inp["sps"],
                                 inp["B_max"], rule)
        assert (got["sel_len"] == ref["sel_len"]).all() and got["objective"][0] == ref["objective"]
    c = np.array([[0.5, 1.0]], np.float32)                     # two peaks: f = 1, 0.9, 1.2
    got = _gpu_schedule_rule(sv, c, [2], np.array([0.0, 1.0, 0.6, 0.6]), 3, sv.SV_STOP_ARGMAX)
    assert int(got["total_rows"][0]) == 3 and list(got["sel_len"]) == [2]
    c1 = np.array([[1.0]], np.float32)                         # tie f(0) = f(1): the smaller b
    got = _gpu_schedule_rule(sv, c1, [1], np.array([0.0, 1.0, 0.5]), 2, sv.SV_STOP_ARGMAX)
    assert int(got["total_rows"][0]) == 1
    got = _gpu_schedule_rule(sv, c1, [0], np.array([0.0, 1.0, 0.5]), 2, sv.SV_STOP_ARGMAX)
    assert int(got["total_rows"][0]) == 1                      # nothing extendable


def test_acceptance_update_matches_oracle(sv, orc):
    """Several rounds with decay and a Beta(2, 3) prior: counts and estimates bit-exact, the
    estimates broadcast to every request's row, and a bad round reported."""
    rng = np.random.default_rng(31)
    N, K = 777, 13
    t_ref, a_ref = np.zeros(K), np.zeros(K)
    t_dev = torch.zeros(K, dtype=torch.float64, device="cuda")
    a_dev = torch.zeros(K, dtype=torch.float64, device="cuda")
    cond = torch.empty((N, K), dtype=torch.float32, device="cuda")
    for rnd in range(4):
        sel = rng.integers(0, K + 1, N).astype(np.int32)
        acc = np.minimum(rng.geometric(0.3, N) - 1, sel).astype(np.int32)
        st, alpha = orc.acceptance_update(sel, acc, K, t_ref, a_ref, decay=0.9, prior_a=2.0,
                                          prior_b=3.0)
        assert st == 0
        out = sv.dspark_acceptance_update(torch.from_numpy(sel).cuda(), torch.from_numpy(acc).cuda(),
                                          t_dev, a_dev, decay=0.9, prior_a=2.0, prior_b=3.0,
                                          cond_accept_out=cond)
        torch.cuda.synchronize()
        assert int(out["status"].item()) == 0
        assert (t_dev.cpu().numpy() == t_ref).all() and (a_dev.cpu().numpy() == a_ref).all()
        assert (out["alpha"].cpu().numpy().view(np.uint32) == alpha.view(np.uint32)).all()
        assert (cond.cpu().numpy() == alpha[None, :]).all()
    bad_sel = torch.tensor([2, 1], dtype=torch.int32, device="cuda")
    bad_acc = torch.tensor([1, 2], dtype=torch.int32, device="cuda")  # accepted > verified
    out = sv.dspark_acceptance_update(bad_sel, bad_acc, t_dev[:2].clone(), a_dev[:2].clone())
    torch.cuda.synchronize()
    assert int(out["status"].item()) == sv.SV_ERR_BAD_INPUT


def test_adaptive_round_on_device(sv, orc):
    """Learned acceptance -> best-budget schedule -> token verification -> acceptance update,
    chained on the device with no host round trip, against the same chain in the oracle."""
    N, K = 48, 8
    rng = np.random.default_rng(5)
    # a previous round's outcome seeds the counts (the drafter has no confidence head)
    sel0 = np.full(N, K, np.int32)
    acc0 = np.minimum(rng.geometric(0.25, N) - 1, K).astype(np.int32)
    t_ref, a_ref = np.zeros(K), np.zeros(K)
    _, alpha = orc.acceptance_update(sel0, acc0, K, t_ref, a_ref)
    cond_ref = np.repeat(alpha[None, :], N, axis=0)
    B_max = N * (K + 1)
    sps = 1.0 / (2e-3 + np.arange(B_max + 1) * 2e-5)
    ref_s = orc.schedule(cond_ref, np.full(N, K, np.int32), sps, B_max, rule=orc.STOP_ARGMAX)
    vw = synth.scaled(synth.SCHEDULED_VERIFY, B=N, gamma=K, V=20000)
    vin = synth.token_inputs(vw, device="cpu")
    tokens = oracle_tokens(orc, vin)
    vref_in = dict(vin, draft_len=torch.from_numpy(ref_s["sel_len"]))
    ref_v = oracle_verify(orc, 0, vref_in, tokens)
    st, alpha1 = orc.acceptance_update(ref_s["sel_len"], ref_v["accepted_len"], K, t_ref, a_ref)
    assert st == 0

    t_dev = torch.zeros(K, dtype=torch.float64, device="cuda")
    a_dev = torch.zeros(K, dtype=torch.float64, device="cuda")
    cond = torch.empty((N, K), dtype=torch.float32, device="cuda")
    sv.dspark_acceptance_update(torch.from_numpy(sel0).cuda(), torch.from_numpy(acc0).cuda(),
                                t_dev, a_dev, cond_accept_out=cond)
    sched = sv.dspark_schedule(cond, torch.full((N,), K, dtype=torch.int32, device="cuda"),
                               torch.from_numpy(sps).cuda(), B_max, rule=sv.SV_STOP_ARGMAX)
    d = {k: vin[k].cuda() for k in ("target", "draft", "target_row0", "draft_row0")}
    ver = sv.spec_verify_token(d["target"], d["draft"], d["target_row0"], d["draft_row0"],
                               sched["sel_len"], K, torch.from_numpy(tokens).cuda(), vin["seed"])
    upd = sv.dspark_acceptance_update(sched["sel_len"], ver["accepted_len"], t_dev, a_dev)
    torch.cuda.synchronize()
    assert int(ver["status"].item()) == 0 and int(upd["status"].item()) == 0
    assert (sched["sel_len"].cpu().numpy() == ref_s["sel_len"]).all()
    lay = layout_np(vref_in)
    res = compare_verify(ver, ref_v, 0, lay["draft_len"], lay["draft_row0"])
    if res["exempt_mismatch"] == 0:
        assert (t_dev.cpu().numpy() == t_ref).all() and (a_dev.cpu().numpy() == a_ref).all()
        assert (upd["alpha"].cpu().numpy() == alpha1).all()
    print(f"\n[parity] adaptive round: {res}")


def test_scheduled_round_full_size(sv, orc):
    """The benchmark's scheduled round at full size: the device schedule of the 512 x 16
    workload feeds token-level verification of V = 129280 bf16 rows laid out as the benchmark
    lays them out (17 target and 16 draft rows per request, only the selected prefixes read), and
    every request is compared with the oracle.  The oracle gets the selected rows only and runs
    on all host threads (its C calls release the interpreter lock)."""
    import concurrent.futures as cf
    import os
    sw = synth.SCHEDULE
    si = synth.schedule_inputs(sw)
    vw = synth.SCHEDULED_VERIFY
    B, G, V = vw.B, vw.gamma, vw.V
    vin = synth.token_inputs(vw, device="cuda")
    sched = sv.dspark_schedule(torch.from_numpy(si["cond_accept"]).cuda(),
                               torch.from_numpy(si["max_len"]).cuda(),
                               torch.from_numpy(si["sps"]).cuda(), si["B_max"])
    ref_s = orc.schedule(si["cond_accept"], si["max_len"], si["sps"], si["B_max"])
    torch.cuda.synchronize()
    sel = ref_s["sel_len"].astype(np.int32)
    assert (sched["sel_len"].cpu().numpy() == sel).all()
    # compact host copies of exactly the rows the verifier reads
    t_rows = np.concatenate([np.arange(r * (G + 1), r * (G + 1) + sel[r] + 1) for r in range(B)])
    d_rows = np.concatenate([np.arange(r * G, r * G + sel[r]) for r in range(B)])
    tgt = vin["target"][torch.from_numpy(t_rows).cuda()].float().cpu().numpy()
    drf = vin["draft"][torch.from_numpy(d_rows).cuda()].float().cpu().numpy()
    t0 = np.concatenate([[0], np.cumsum(sel + 1)[:-1]]).astype(np.int64)
    d0 = np.concatenate([[0], np.cumsum(sel)[:-1]]).astype(np.int64)
    workers = os.cpu_count() or 1
    chunks = [(a, min(B, a + 16)) for a in range(0, B, 16)]

    def sample(ch):
        a, b = ch
        st, tok = orc.sample_draft_batch(drf, V, V, d0[a:b], sel[a:b], b - a, vw.seed,
                                         request_ids=np.arange(a, b, dtype=np.uint64),
                                         n_draft_rows=drf.shape[0])
        assert st == 0
        return tok
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        parts = list(ex.map(sample, chunks))
    tok_c = np.max(np.stack(parts), axis=0).astype(np.int32)  # each row filled by one chunk
    assert (tok_c >= 0).all()

    def verify(ch):
        a, b = ch
        return orc.verify_batch(0, tgt, drf, V, V, t0[a:b], d0[a:b], sel[a:b], tok_c, b - a,
                                vw.seed, request_ids=np.arange(a, b, dtype=np.uint64),
                                out_ld=G + 1)
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        vparts = list(ex.map(verify, chunks))
    assert all(p["status"] == 0 for p in vparts)
    ref = {k: np.concatenate([p[k] for p in vparts])
           for k in ("accepted_len", "out_tokens", "decision_margin", "race_margin")}
    ratio = np.full(B * G, np.nan)
    for (a, b), p in zip(chunks, vparts):
        for r in range(a, b):
            ratio[r * G: r * G + sel[r]] = p["ratio"][d0[r]: d0[r] + sel[r]]
    ref["ratio"] = ratio
    # the device chain: scheduler lengths straight into the verifier, full row layout
    tokens = np.zeros(B * G, np.int32)
    tokens[d_rows] = tok_c
    gpu = sv.spec_verify_token(vin["target"], vin["draft"], vin["target_row0"],
                               vin["draft_row0"], sched["sel_len"], G,
                               torch.from_numpy(tokens).cuda(), vw.seed)
    torch.cuda.synchronize()
    assert int(gpu["status"].item()) == 0
    res = compare_verify(gpu, ref, 0, sel, np.arange(B, dtype=np.int64) * G)
    print(f"\n[parity] scheduled round, 512 x 16, V = {V}: {res}, "
          f"{int(sel.sum())} drafted positions verified")
    assert res["requests"] == B


def test_schedule_async_two_stream_chain(sv, orc):
    """Six rounds of the asynchronous scheduler on the device.  A "draft" stream writes each
    round's confidence-head predictions into slot t % 3 of a ring; a "schedule" stream schedules
    round t from slot (t - 2) % 3, waiting only for round t - 2's write (and the draft stream
    overwrites a slot only after the schedule that reads it).  Every round's selection, total and
    objective equal the oracle's chain bit for bit."""
    rng = np.random.default_rng(23)
    N, K, T, depth = 96, 8, 6, 3
    conf = (rng.beta(8, 2, (T, N, K)) * 0.97 ** np.arange(K)).astype(np.float32)
    prior = np.full((N, K), 0.75, np.float32)
    ml = rng.integers(0, K + 1, N).astype(np.int32)
    B_max = N * (K + 1)
    sps = 1.0 / (2e-3 + np.arange(B_max + 1) * 4e-6)
    dev = torch.device("cuda")
    ring = torch.zeros((depth, N, K), dtype=torch.float32, device=dev)
    host = torch.from_numpy(conf).pin_memory()
    prior_d = torch.from_numpy(prior).to(dev)
    ml_d = torch.from_numpy(ml).to(dev)
    sps_d = torch.from_numpy(sps).to(dev)
    torch.cuda.synchronize()
    s_draft, s_sched = torch.cuda.Stream(), torch.cuda.Stream()
    written = [torch.cuda.Event() for _ in range(T)]
    read = [torch.cuda.Event() for _ in range(T)]
    outs = []
    for t in range(T):
        with torch.cuda.stream(s_draft):
            if t >= depth:  # slot t % 3 was last read by the schedule of round t - 1
                s_draft.wait_event(read[t - 1])
            ring[t % depth].copy_(host[t], non_blocking=True)
            written[t].record(s_draft)
        with torch.cuda.stream(s_sched):
            if t >= 2:
                s_sched.wait_event(written[t - 2])
            outs.append(sv.dspark_schedule_async(ring, t, prior_d, ml_d, sps_d, B_max,
                                                 stream=s_sched))
            read[t].record(s_sched)
    torch.cuda.synchronize()
    for t, o in enumerate(outs):
        ref = orc.schedule_async(conf, t, prior, ml, sps, B_max)
        assert ref["status"] == 0 and int(o["status"].item()) == 0
        assert (o["sel_len"].cpu().numpy() == ref["sel_len"]).all(), t
        assert int(o["total_rows"].item()) == ref["total_rows"]
        assert float(o["objective"].item()) == ref["objective"]
    # the selections change from round to round: the chain really reads different slots
    assert len({tuple(o["sel_len"].cpu().numpy()) for o in outs[2:]}) > 1
