"""GPU parity of spec_verify_token / spec_verify_block / spec_sample_draft with the CPU oracle.

Every case feeds both sides the same seeded synthetic logits (synth) and the same drafted tokens
(sampled from q by the oracle); the CUDA path is reached through the C ABI (ctypes binding)."""
import numpy as np
import pytest
import torch

from parity import compare_verify, host_f32, layout_np, oracle_tokens, oracle_verify
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


def _to_dev(inp):
    d = dict(inp)
    for k in ("target", "draft", "target_row0", "draft_row0", "draft_len"):
        d[k] = inp[k].cuda()
    return d


def _run(sv, block, inp, tokens, request_ids=None, want_rows=True):
    """want_rows=False leaves out the per-row outputs; block verification then computes the
    residual mass only for positions whose uniform does not exceed the running ratio."""
    if block:
        out = sv.spec_verify_block(inp["target"], inp["draft"], inp["target_row0"],
                                   inp["draft_row0"], inp["draft_len"], inp["max_draft_len"],
                                   torch.from_numpy(tokens).cuda(), inp["seed"],
                                   request_ids=request_ids, want_rows=want_rows)
    else:
        out = sv.spec_verify_token(inp["target"], inp["draft"], inp["target_row0"],
                                   inp["draft_row0"], inp["draft_len"], inp["max_draft_len"],
                                   torch.from_numpy(tokens).cuda(), inp["seed"],
                                   request_ids=request_ids, want_ratio=want_rows)
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 0, sv.status_string(int(out["status"].item()))
    return out


def _parity(sv, orc, block, inp, tokens=None, request_ids=None, want_rows=True):
    if tokens is None:
        tokens = oracle_tokens(orc, inp)
    rid_np = None if request_ids is None else request_ids.cpu().numpy()
    ref = oracle_verify(orc, block, inp, tokens, request_ids=rid_np)
    assert ref["status"] == 0
    gpu = _run(sv, block, inp, tokens, request_ids, want_rows=want_rows)
    lay = layout_np(inp)
    res = compare_verify(gpu, ref, block, lay["draft_len"], lay["draft_row0"])
    print(f"\n[parity] block={block} rows={want_rows} B={inp['B']} V={inp['V']}: {res}")
    return gpu, ref, res


@pytest.mark.parametrize("block", [0, 1])
def test_token_small_workload(sv, orc, block):
    """4 requests x 4 drafted positions, V = 1024, fp32, Philox seed 0."""
    inp = _to_dev(synth.token_inputs(synth.TOKEN_SMALL, device="cpu"))
    _parity(sv, orc, block, inp)


@pytest.mark.parametrize("block", [0, 1])
@pytest.mark.parametrize("V", [40000, 40003, 8191, 7])
def test_scaled_bf16_ragged_vocab(sv, orc, block, V):
    """bf16 rows spanning several 16 KB slices with a ragged tail (V not a multiple of 8 uses a
    padded row stride)."""
    w = synth.scaled(synth.TOKEN_LARGE, B=12, V=V)
    _parity(sv, orc, block, _padded_dev(synth.token_inputs(w, device="cpu")))


def _padded_dev(inp):
    """Device copy whose rows are padded to a 16-byte stride (V not a multiple of 8)."""
    V = inp["V"]
    ld = (V + 7) // 8 * 8
    for k in ("target", "draft"):
        buf = torch.zeros((inp[k].shape[0], ld), dtype=inp[k].dtype)
        buf[:, :V] = inp[k]
        inp[k] = buf
    inp = _to_dev(inp)
    inp["target"] = inp["target"][:, :V]
    inp["draft"] = inp["draft"][:, :V]
    return inp


@pytest.mark.parametrize("block", [0, 1])
def test_ragged_lengths_and_scattered_rows(sv, orc, block):
    """Per-request drafted lengths 0..7 and rows of each request placed out of order."""
    w = synth.scaled(synth.BLOCK_LARGE, B=40, V=20000)
    lens = synth.ragged_lengths(40, 7, seed=3)
    inp = synth.token_inputs(w, device="cpu", draft_len=lens)
    perm = torch.from_numpy(np.random.default_rng(4).permutation(40))
    inp["target_row0"] = inp["target_row0"][perm].contiguous()
    inp["draft_row0"] = inp["draft_row0"][perm].contiguous()
    inp = _to_dev(inp)
    rids = torch.from_numpy(np.random.default_rng(5).integers(0, 2**60, 40).astype(np.uint64)
                            .view(np.int64)).cuda()
    _parity(sv, orc, block, inp, request_ids=rids)


@pytest.mark.parametrize("block", [0, 1])
def test_full_size_workloads(sv, orc, block):
    """Token-level: 64 requests x 5 positions, V = 151936 bf16.  Block: 128 requests x 7
    positions, V = 129280 bf16.  Every request compared."""
    w = synth.BLOCK_LARGE if block else synth.TOKEN_LARGE
    inp = _to_dev(synth.token_inputs(w, device="cpu"))
    _parity(sv, orc, block, inp)


@pytest.mark.parametrize("case", ["small_f32", "ragged_vocab", "ragged_lengths", "full_size"])
def test_block_without_row_outputs(sv, orc, case):
    """Block verification without the per-row outputs skips the residual pass of positions whose
    uniform exceeds the running ratio (h_i <= rho_i < eta_i fails whatever R_i is).  Accepted
    lengths and tokens must still equal the oracle's; and, on the same inputs, the call with the
    per-row outputs must agree with it exactly."""
    rids = None
    if case == "small_f32":
        inp = _to_dev(synth.token_inputs(synth.TOKEN_SMALL, device="cpu"))
    elif case == "ragged_vocab":
        inp = _padded_dev(synth.token_inputs(synth.scaled(synth.BLOCK_LARGE, B=24, V=40003),
                                             device="cpu"))
    elif case == "ragged_lengths":
        w = synth.scaled(synth.BLOCK_LARGE, B=40, V=20000)
        inp = synth.token_inputs(w, device="cpu", draft_len=synth.ragged_lengths(40, 7, seed=9))
        inp = _to_dev(inp)
        rids = torch.arange(1000, 1040, dtype=torch.int64).cuda()
    else:
        inp = _to_dev(synth.token_inputs(synth.BLOCK_LARGE, device="cpu"))
    tokens = oracle_tokens(orc, inp)
    gpu, _, _ = _parity(sv, orc, 1, inp, tokens=tokens, request_ids=rids, want_rows=False)
    full = _run(sv, 1, inp, tokens, request_ids=rids, want_rows=True)
    assert torch.equal(gpu["accepted_len"], full["accepted_len"])
    assert torch.equal(gpu["out_tokens"], full["out_tokens"])


@pytest.mark.parametrize("block", [0, 1])
def test_more_requests_than_sms(sv, orc, block):
    """400 requests with ragged lengths: the block kernel's CTAs each walk several requests in
    turn (request numbers, the shared race bound and the decision reused), with and without the
    per-row outputs."""
    w = synth.scaled(synth.BLOCK_LARGE, B=400, V=3000)
    inp = _to_dev(synth.token_inputs(w, device="cpu",
                                     draft_len=synth.ragged_lengths(400, 7, seed=13)))
    tokens = oracle_tokens(orc, inp)
    _parity(sv, orc, block, inp, tokens=tokens)
    if block:
        _parity(sv, orc, block, inp, tokens=tokens, want_rows=False)


@pytest.mark.parametrize("gamma,noise", [(32, 0.02), (32, 1.0), (40, 0.02)])
def test_long_drafts(sv, orc, gamma, noise):
    """Token-level verification of long drafts (32 and 40 positions).  A small draft perturbation
    makes long accepted runs and bonus tokens common, so the decision walks far into the request
    and races the bonus row; lengths are ragged, with some requests at the maximum."""
    w = synth.scaled(synth.TOKEN_LARGE, B=24, gamma=gamma, V=6000, draft_noise=noise)
    lens = synth.ragged_lengths(24, gamma, seed=21)
    lens[:4] = gamma
    inp = _to_dev(synth.token_inputs(w, device="cpu", draft_len=lens))
    gpu, ref, _ = _parity(sv, orc, 0, inp)
    if noise < 0.1:
        assert (ref["accepted_len"] >= 16).sum() >= 4  # long runs were exercised


def test_sampler_matches_oracle(sv, orc):
    """Draft tokens raced from q on the GPU equal the oracle's, except counted near-ties."""
    for w in (synth.TOKEN_SMALL, synth.scaled(synth.TOKEN_LARGE, B=16, V=50000)):
        inp = synth.token_inputs(w, device="cpu")
        ref = oracle_tokens(orc, inp)
        d = _to_dev(inp)
        got = sv.spec_sample_draft(d["draft"], d["draft_row0"], d["draft_len"],
                                   d["max_draft_len"], d["seed"]).cpu().numpy()
        # every mismatch must be a near-tie of the oracle's race, and near ties are rare
        draft = host_f32(inp["draft"])
        miss = np.flatnonzero(got != ref)
        assert miss.size <= max(1, int(np.ceil(0.01 * ref.size))), miss
        for row in miss:
            r, i = divmod(int(row), w.gamma)
            st, tok, margin = orc.sample_race(draft[row], w.seed, r, i + 1, orc.TAG_DRAFT)
            assert tok == ref[row] and margin < 1e-5


def test_determinism(sv, orc):
    inp = _to_dev(synth.token_inputs(synth.scaled(synth.TOKEN_LARGE, B=8, V=30000), "cpu"))
    tokens = oracle_tokens(orc, inp)
    a = _run(sv, 0, inp, tokens)
    b = _run(sv, 0, inp, tokens)
    assert torch.equal(a["out_tokens"], b["out_tokens"])
    assert torch.equal(a["accept_ratio"], b["accept_ratio"])


@pytest.mark.parametrize("block", [0, 1])
def test_all_zero_drafts_and_masked_rows(sv, orc, block):
    """gamma = 0 everywhere (bonus only) and rows with masked (-inf) entries."""
    w = synth.scaled(synth.TOKEN_LARGE, B=6, V=9000)
    inp = synth.token_inputs(w, "cpu", draft_len=np.zeros(6, np.int32))
    inp["target"][:, :4000] = float("-inf")
    inp = _to_dev(inp)
    gpu, ref, _ = _parity(sv, orc, block, inp,
                          tokens=np.zeros(inp["draft"].shape[0], np.int32))
    assert (gpu["correction"].cpu().numpy() >= 4000).all()


@pytest.mark.parametrize("block", [0, 1])
def test_data_errors_reported(sv, orc, block):
    w = synth.scaled(synth.TOKEN_SMALL, B=2)
    base = synth.token_inputs(w, "cpu")
    tokens = oracle_tokens(orc, base)
    cases = []
    bad_tok = tokens.copy()
    bad_tok[1] = w.V + 3
    cases.append((base, bad_tok))
    nan_in = dict(base, target=base["target"].clone())
    nan_in["target"][2, 5] = float("nan")
    cases.append((nan_in, tokens))
    zq = dict(base, draft=base["draft"].clone())
    zq["draft"][0, int(tokens[0])] = float("-inf")
    cases.append((zq, tokens))
    bad_len = dict(base, draft_len=torch.tensor([2, w.gamma + 1], dtype=torch.int32))
    cases.append((bad_len, tokens))
    for inp, toks in cases:
        d = _to_dev(inp)
        fn = sv.spec_verify_block if block else sv.spec_verify_token
        out = fn(d["target"], d["draft"], d["target_row0"], d["draft_row0"], d["draft_len"],
                 d["max_draft_len"], torch.from_numpy(toks).cuda(), d["seed"])
        torch.cuda.synchronize()
        assert int(out["status"].item()) == sv.SV_ERR_BAD_INPUT


def test_empty_batch_and_argument_errors(sv):
    z = torch.zeros((1, 1024), device="cuda")
    i64 = torch.zeros(0, dtype=torch.int64, device="cuda")
    i32 = torch.zeros(0, dtype=torch.int32, device="cuda")
    out = sv.spec_verify_token(z, z, i64, i64, i32, 4, torch.zeros(1, dtype=torch.int32,
                                                                    device="cuda"), 0)
    assert out["accepted_len"].numel() == 0
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_token(z, z, i64, i64, i32, sv.SV_MAX_DRAFT_LEN + 1,
                             torch.zeros(1, dtype=torch.int32, device="cuda"), 0)


def _residual_empty_batch(orc, B, gamma, V, dtype, seed):
    """Requests whose correction residual is empty to working precision on both sides.

    Request r % 3 == 0: position 1 is degenerate -- the target masks the drafted token x
    (p(x) = 0) and the draft gives it the logit -120 (weight ~e^-120, lost when added to a
    normaliser of order one in binary32 and binary64), every other entry equal in both rows; so
    p(x)/q(x) = 0 rejects x and max(p - q, 0) is empty.  Request r % 3 == 1: position 1 has equal
    target and draft rows (ratio exactly 1, always accepted; for block verification R_1 = 0 and
    R_1 + 1 - rho_1 = 0, so h_1 = 1) and position 2 is degenerate.  Request r % 3 == 2: ordinary
    rows.  Returns the inputs, the drafted tokens and the requests expected to fall back."""
    w = synth.scaled(synth.TOKEN_LARGE, B=B, gamma=gamma, V=V, dtype=dtype)
    inp = synth.token_inputs(w, device="cpu")
    tokens = oracle_tokens(orc, inp)
    rng = np.random.default_rng(seed)
    t, d = inp["target"], inp["draft"]
    fall = []
    for r in range(B):
        kind = r % 3
        if kind == 2:
            continue
        pos = 1 if kind == 0 else 2
        if kind == 1:
            d[r * gamma] = t[r * (gamma + 1)]  # position 1: draft row = target row
        trow, drow = r * (gamma + 1) + pos - 1, r * gamma + pos - 1
        x = int(rng.integers(V // 2, V))
        d[drow] = t[trow]
        t[trow, x] = float("-inf")
        d[drow, x] = -120.0
        tokens[drow] = x
        fall.append(r)
    return inp, tokens, np.array(fall)


@pytest.mark.parametrize("block", [0, 1])
@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 20000), (torch.float32, 4099)])
def test_residual_empty_fallback(sv, orc, block, dtype, V):
    """An empty residual at the first rejection: both sides draw the correction from p with the
    RESID uniforms of that position (the oracle reports the fallback), token for token."""
    inp, tokens, fall = _residual_empty_batch(orc, 12, 3, V, dtype, seed=17)
    dev = _padded_dev(inp) if (V * inp["target"].element_size()) % 16 else _to_dev(inp)
    gpu, ref, res = _parity(sv, orc, block, dev, tokens=tokens)
    kinds = ref["race_kind"]
    assert (kinds[fall] == orc.RACE_RESIDUAL_EMPTY).all(), kinds
    assert (ref["accepted_len"][fall] == fall % 3).all()
    assert res["exempt_mismatch"] == 0


@pytest.mark.parametrize("block", [0, 1])
def test_gpu_emitted_histogram_chisquare_1e6(sv, block):
    """10^6 independent requests on V = 4, gamma = 2 (fp32), drafts drawn from q by the library's
    sampler and verified on the GPU: the first emitted token follows p_1 (chi-square, 3 degrees of
    freedom, the 1e-4 critical value) -- the distribution itself, beside the request-by-request
    parity with the oracle."""
    from scipy.special import softmax
    from scipy.stats import chi2, chisquare
    V, G, n = 4, 2, 1_000_000
    rng = np.random.default_rng(2025)
    T = rng.normal(0, 1.0, (G + 1, V)).astype(np.float32)
    D = (T[:G] + rng.normal(0, 0.8, (G, V))).astype(np.float32)
    tgt = torch.from_numpy(np.tile(T, (n, 1))).cuda()
    drf = torch.from_numpy(np.tile(D, (n, 1))).cuda()
    tr0 = torch.arange(n, dtype=torch.int64, device="cuda") * (G + 1)
    dr0 = torch.arange(n, dtype=torch.int64, device="cuda") * G
    dl = torch.full((n,), G, dtype=torch.int32, device="cuda")
    toks = sv.spec_sample_draft(drf, dr0, dl, G, 19)
    fn = sv.spec_verify_block if block else sv.spec_verify_token
    out = fn(tgt, drf, tr0, dr0, dl, G, toks, 19)
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 0
    counts = np.bincount(out["out_tokens"][:, 0].cpu().numpy(), minlength=V)
    stat = chisquare(counts, n * softmax(T[0].astype(np.float64))).statistic
    assert stat < chi2.ppf(1 - 1e-4, V - 1), (counts, stat)


@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 3001), (torch.float32, 2999)])
def test_flat_rows_sample_the_largest_race_uniform(sv, orc, dtype, V):
    """Rows of equal logits: every key is one constant plus the noise of its race uniform, so the
    sampler must return the entry of largest uniform -- the oracle's race_uniform, evaluated entry
    by entry -- for each drafted row.  Exercises the coarse-half gate where every entry is within
    reach of the bound, the FINE blocks, the ragged tail (V not a multiple of 8) and request ids
    with high bits."""
    B, G, seed = 5, 3, 2024
    rids = np.array([7, 2**33 + 1, 2**47 + 12345, 0, 99], dtype=np.uint64)
    ld = (V + 7) // 8 * 8  # row starts 16-byte aligned
    drf = torch.zeros((B * G, ld), dtype=dtype, device="cuda")[:, :V]
    dr0 = torch.arange(B, dtype=torch.int64, device="cuda") * G
    dl = torch.full((B,), G, dtype=torch.int32, device="cuda")
    toks = sv.spec_sample_draft(drf, dr0, dl, G, seed,
                                request_ids=torch.from_numpy(rids.view(np.int64)).cuda())
    torch.cuda.synchronize()
    toks = toks.cpu().numpy()
    for r in range(B):
        for i in range(G):
            u = np.array([orc.race_uniform(seed, int(rids[r]), i + 1, orc.TAG_DRAFT, v)
                          for v in range(V)])
            assert toks[r * G + i] == int(np.argmax(u)), (r, i)
